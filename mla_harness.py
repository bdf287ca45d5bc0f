"""Device-side set-up for tests, the benchmark and the smoke check.

Uploads a drawn workload (mla_inputs.Problem) to the GPU, lays out the paged
cache and runs one decode step through the library's C ABI.  Contains no
attention arithmetic of its own.
"""
from __future__ import annotations

import numpy as np
import torch

import mla_inputs as I
import mla_latent_kv_81_b300 as M


def tdtype(dtype: str):
    return torch.bfloat16 if dtype == "bf16" else torch.float32


def to_dev(a: np.ndarray, dtype: str, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=tdtype(dtype))


class DeviceLayer:
    """One MLA layer's weights, paged cache and RoPE table on the device."""

    fp8 = False   # reduced-precision cache (set per workload in __init__)

    def __init__(self, p: I.Problem, device="cuda", max_pos: int | None = None):
        self.p = p
        w, d = p.w, p.dims
        self.device = device
        self.dt = tdtype(w.dtype)
        self.fp8 = bool(getattr(w, "cache_fp8", False))
        self.cfg = M.make_config(d, w.dtype, cache_fp8=self.fp8)
        self.W = {k: to_dev(v, w.dtype, device) for k, v in p.weights.items()}
        if self.fp8:
            # reduced-precision blocks as raw bytes: codes [d_c][bs], k_R / s [d_rope][bs] bf16, s [bs] fp32;
            # 0xFF everywhere unwritten (a NaN code, a NaN bf16, a NaN scale)
            self.fp8_block_bytes = d.block_size * (d.d_c + 2 * d.d_rope + 4)
            self.pool = torch.full((p.num_blocks, self.fp8_block_bytes), 255, dtype=torch.uint8, device=device)
        else:
            # each block stored transposed: [row element][block_size tokens]; NaN sentinels everywhere unwritten
            self.pool = torch.full((p.num_blocks, d.row, d.block_size), float("nan"), dtype=self.dt, device=device)
        self.block_table = torch.from_numpy(p.block_table).to(device)
        if max_pos is None:
            max_pos = int(p.block_table.shape[1]) * d.block_size + 8
        self.rope_tab = torch.empty((max_pos, d.d_rope // 2, 2), dtype=torch.float32, device=device)
        M.mla_rope_table_create(self.cfg, d.rope_base, max_pos, self.rope_tab)
        self.rope = M.make_rope(self.rope_tab)
        self.cache = M.make_cache(self.pool, self.block_table, d.block_size)
        self.kv_len = torch.from_numpy(p.kv_len.astype(np.int32)).to(device)
        self.x_q = to_dev(p.x_q, w.dtype, device)
        self.q_pos = torch.from_numpy(p.q_pos).to(device)
        n = p.w.batch * p.w.n_q
        self.q = torch.empty((n, d.n_heads, d.row), dtype=self.dt, device=device)
        self.o_lat = torch.empty((n, d.n_heads, d.d_c), dtype=self.dt, device=device)
        self.lse = torch.empty((n, d.n_heads), dtype=torch.float32, device=device)
        self.out = torch.empty((n, d.d_model), dtype=self.dt, device=device)
        # the query tokens appended before attention (their hidden states are the queries)
        if p.w.n_append:
            self.app_seq = torch.from_numpy(np.repeat(np.arange(p.w.batch), p.w.n_q).astype(np.int32)).to(device)
            self.app_pos = self.q_pos
        self.ws = {}

    # ---------------------------------------------------------------- cache fill
    def fp8_parts(self):
        """Views of the reduced-precision pool: codes [nb, d_c, bs] uint8, k_R / s [nb, d_rope, bs] bf16,
        s [nb, bs] fp32."""
        d = self.p.dims
        bs, nb = d.block_size, self.pool.shape[0]
        codes = self.pool[:, :d.d_c * bs].view(nb, d.d_c, bs)
        kr = self.pool[:, d.d_c * bs:(d.d_c + 2 * d.d_rope) * bs].view(torch.bfloat16).view(nb, d.d_rope, bs)
        sc = self.pool[:, (d.d_c + 2 * d.d_rope) * bs:].view(torch.float32).view(nb, bs)
        return codes, kr, sc

    def fill_direct(self):
        """Write drawn latent rows at every cached position (no projection involved)."""
        p, d = self.p, self.p.dims
        bs = d.block_size
        if self.fp8:
            codes_v, kr_v, sc_v = self.fp8_parts()
            for b in range(p.w.batch):
                L = int(p.lens[b])
                if L == 0:
                    continue
                codes, k, kr = I.draw_fp8_rows(p.w, b, L)
                pos = np.arange(L)
                blk = torch.from_numpy(p.block_table[b, pos // bs].astype(np.int64)).to(self.device)
                off = torch.from_numpy(pos % bs).to(self.device)
                codes_v[blk, :, off] = torch.from_numpy(codes).to(self.device)
                kr_v[blk, :, off] = torch.from_numpy(kr).to(self.device, torch.bfloat16)
                sc_v[blk, off] = torch.from_numpy(np.ldexp(np.float32(1.0), k).astype(np.float32)).to(self.device)
            return
        for b in range(p.w.batch):
            L = int(p.lens[b])
            if L == 0:
                continue
            rows = to_dev(I.draw_latent_rows(p.w, b, L), p.w.dtype, self.device)
            n_full = L // bs
            if n_full:
                blks = torch.from_numpy(p.block_table[b, :n_full].astype(np.int64)).to(self.device)
                self.pool[blks] = rows[:n_full * bs].reshape(n_full, bs, d.row).transpose(1, 2)
            rem = L - n_full * bs
            if rem:
                self.pool[int(p.block_table[b, n_full]), :, :rem] = rows[n_full * bs:].T

    def fill_by_append(self, chunk: int = 8192):
        """Build the cache from x_ctx with mla_compress_append (positions 0..L_b-1)."""
        p = self.p
        seq = np.repeat(np.arange(p.w.batch), p.lens).astype(np.int32)
        pos = np.concatenate([np.arange(L) for L in p.lens]).astype(np.int32)
        for s in range(0, len(seq), chunk):
            x = to_dev(p.x_ctx[s:s + chunk], p.w.dtype, self.device)
            ws = self._ws("fill", M.mla_compress_workspace_bytes(self.cfg, x.shape[0]))
            M.mla_compress_append(self.cfg, x, self.W["W_DKV"], self.W["W_KR"],
                                  torch.from_numpy(seq[s:s + chunk]).to(self.device),
                                  torch.from_numpy(pos[s:s + chunk]).to(self.device), self.rope, self.cache, ws=ws)

    def fill(self):
        if self.p.w.fill == "direct":
            self.fill_direct()
        else:
            self.fill_by_append()

    # ---------------------------------------------------------------- one decode step
    def _ws(self, key, nbytes):
        t = self.ws.get(key)
        if t is None or t.numel() < nbytes:
            if t is not None:
                # keep the flags the old workspace collected
                code, flags = M.mla_get_device_status(t)
                self.carried_flags = getattr(self, "carried_flags", 0) | flags
            t = M.workspace(nbytes, self.device)
            self.ws[key] = t
        return t

    def status(self, stream=None):
        """(code, flags) over every workspace this layer's calls used (and clears them): the OR of their
        status words; code is MLA_ERR_DEVICE_INDEX (5) if any index flag, MLA_ERR_TIMEOUT (4) if any
        timeout, else 0."""
        flags = getattr(self, "carried_flags", 0)
        self.carried_flags = 0
        for t in self.ws.values():
            _, f = M.mla_get_device_status(t, stream)
            flags |= f
        return (5 if flags & 1 else 4 if flags & 2 else 0), flags

    def step(self, x_q=None, stream=None, with_lse=True):
        p, cfg = self.p, self.cfg
        x_q = self.x_q if x_q is None else x_q
        n = x_q.shape[0]
        if p.w.n_append:
            ws = self._ws("c", M.mla_compress_workspace_bytes(cfg, n))
            M.mla_compress_append(cfg, x_q, self.W["W_DKV"], self.W["W_KR"], self.app_seq, self.app_pos, self.rope,
                                  self.cache, ws=ws, stream=stream)
        ws = self._ws("a", M.mla_absorb_workspace_bytes(cfg, n))
        M.mla_absorb_query(cfg, x_q, self.W["W_Q"], self.W["W_QR"], self.W["W_UK"], self.q_pos, self.rope, self.q,
                           ws=ws, stream=stream)
        self.attend(stream=stream, with_lse=with_lse)
        ws = self._ws("o", M.mla_output_workspace_bytes(cfg, n))
        M.mla_output_project(cfg, self.o_lat, self.W["W_UV"], self.W["W_O"], self.out, ws=ws, stream=stream)
        return self.out

    def attend(self, q=None, stream=None, with_lse=True):
        p = self.p
        ws = self._ws("d", M.mla_decode_workspace_bytes(self.cfg, p.w.batch, p.w.n_q, self.cache.max_blocks_per_seq))
        M.mla_decode_attention(self.cfg, self.q if q is None else q, self.cache, self.kv_len, p.w.batch, p.w.n_q,
                               self.o_lat, self.lse if with_lse else None, ws=ws, stream=stream)
        return self.o_lat

    # ---------------------------------------------------------------- host copies for the oracle
    def pool_token_bits(self) -> np.ndarray:
        """Raw bit patterns of the whole pool as [num_blocks, block_size, row] (int16 for bf16, int32 for fp32)."""
        raw = self.pool.view(torch.int16 if self.p.w.dtype == "bf16" else torch.int32)
        return raw.transpose(1, 2).cpu().numpy()

    def cache_rows_at(self, seq, pos) -> np.ndarray:
        """Rows at logical positions pos[i] of sequences seq[i], read back from the pool (float32 numpy).
        For a reduced-precision pool: (codes uint8 [n, d_c], k_R / s float32 [n, d_rope], s float32 [n])."""
        bs = self.p.dims.block_size
        seq, pos = np.asarray(seq, dtype=np.int64), np.asarray(pos, dtype=np.int64)
        blk = torch.from_numpy(self.p.block_table[seq, pos // bs].astype(np.int64)).to(self.device)
        off = torch.from_numpy(pos % bs).to(self.device)
        if self.fp8:
            codes, kr, sc = self.fp8_parts()
            return (codes[blk, :, off].cpu().numpy(), kr[blk, :, off].float().cpu().numpy(),
                    sc[blk, off].cpu().numpy())
        return self.pool[blk, :, off].float().cpu().numpy()

    def cache_rows_logical(self, b: int, n: int | None = None) -> np.ndarray:
        """Rows 0..n-1 of sequence b read back from the pool, as float32 numpy (exact bf16 values)."""
        n = int(self.p.kv_len[b]) if n is None else n
        return self.cache_rows_at(np.full(n, b), np.arange(n))


def write_rows(pool, block_table: np.ndarray, b: int, rows, block_size: int):
    """Store token-major rows [n, row] at positions 0..n-1 of sequence b of an element-major pool."""
    n = rows.shape[0]
    n_full = n // block_size
    if n_full:
        blks = torch.from_numpy(block_table[b, :n_full].astype(np.int64)).to(pool.device)
        pool[blks] = rows[:n_full * block_size].reshape(n_full, block_size, rows.shape[1]).transpose(1, 2)
    rem = n - n_full * block_size
    if rem:
        pool[int(block_table[b, n_full]), :, :rem] = rows[n_full * block_size:].T


class PrefillLayer:
    """A prompt on the device (mla_inputs.PrefillProblem) and the explicit-form calls over it."""

    def __init__(self, p: I.PrefillProblem, device="cuda"):
        self.p = p
        c, d = p.case, p.dims
        self.device = device
        self.dt = tdtype(c.dtype)
        self.cfg = M.make_config(d, c.dtype, cache_fp8=c.cache_fp8, rope_per_head=c.rope_per_head)
        self.W = {k: to_dev(v, c.dtype, device) for k, v in p.weights.items()}
        row = d.d_c + (d.n_heads if c.rope_per_head else 1) * d.d_rope
        if c.cache_fp8:
            self.pool = torch.full((p.num_blocks, d.block_size * (d.d_c + 2 * d.d_rope + 4)), 255, dtype=torch.uint8,
                                   device=device)
        else:
            self.pool = torch.full((p.num_blocks, row, d.block_size), float("nan"), dtype=self.dt, device=device)
        self.block_table = torch.from_numpy(p.block_table).to(device)
        self.cache = M.make_cache(self.pool, self.block_table, d.block_size)
        max_pos = int(p.block_table.shape[1]) * d.block_size + 8
        self.rope_tab = torch.empty((max_pos, d.d_rope // 2, 2), dtype=torch.float32, device=device)
        M.mla_rope_table_create(self.cfg, d.rope_base, max_pos, self.rope_tab)
        self.rope = M.make_rope(self.rope_tab)
        T = c.queries
        self.q = (to_dev(p.q, c.dtype, device) if p.q is not None else
                  torch.empty((T, d.n_heads, d.qk_nope + d.d_rope), dtype=self.dt, device=device))
        self.o = torch.empty((T, d.n_heads, d.v_head), dtype=self.dt, device=device)
        self.lse = torch.empty((T, d.n_heads), dtype=torch.float32, device=device)
        self.out = torch.empty((T, d.d_model), dtype=self.dt, device=device)
        self.ws = {}
        if p.x is not None:
            self.x = to_dev(p.x, c.dtype, device)

    def _ws(self, key, nbytes):
        t = self.ws.get(key)
        if t is None or t.numel() < nbytes:
            t = M.workspace(nbytes, self.device)
            self.ws[key] = t
        return t

    def status(self, stream=None):
        flags = 0
        for t in self.ws.values():
            _, f = M.mla_get_device_status(t, stream)
            flags |= f
        return (5 if flags & 1 else 4 if flags & 2 else 0), flags

    def fill(self):
        """Cache rows of the prompt: drawn rows written directly, or appended from the hidden states."""
        p, c, d = self.p, self.p.case, self.p.dims
        if p.rows is not None:
            write_rows(self.pool, p.block_table, c.seq, to_dev(p.rows, c.dtype, self.device), d.block_size)
            return
        L = c.prompt
        seq = torch.full((L,), c.seq, dtype=torch.int32, device=self.device)
        pos = torch.arange(L, dtype=torch.int32, device=self.device)
        ws = self._ws("fill", M.mla_compress_workspace_bytes(self.cfg, L))
        M.mla_compress_append(self.cfg, self.x, self.W["W_DKV"], self.W["W_KR"], seq, pos, self.rope, self.cache,
                              ws=ws)

    def project(self, stream=None):
        """Queries [q_nope || q_R] of the last `queries` prompt tokens from their hidden states."""
        c = self.p.case
        xq = self.x[c.prompt - c.queries:]
        q_pos = torch.from_numpy(self.p.q_pos).to(self.device)
        ws = self._ws("q", M.mla_project_workspace_bytes(self.cfg, c.queries))
        M.mla_project_query(self.cfg, xq, self.W["W_Q"], self.W["W_QR"], q_pos, self.rope, self.q, ws=ws,
                            stream=stream)
        return self.q

    def attend(self, stream=None, with_lse=True):
        c = self.p.case
        ws = self._ws("p", M.mla_prefill_workspace_bytes(self.cfg, c.prompt))
        M.mla_prefill_attention(self.cfg, self.q, self.cache, c.seq, c.prompt, self.W["W_UK"], self.W["W_UV"],
                                self.o, self.lse if with_lse else None, ws=ws, stream=stream)
        return self.o

    def output(self, stream=None):
        ws = self._ws("o", M.mla_head_output_workspace_bytes(self.cfg, self.p.case.queries))
        M.mla_head_output_project(self.cfg, self.o, self.W["W_O"], self.out, ws=ws, stream=stream)
        return self.out

    def run(self, stream=None):
        """The explicit-form layer from hidden states: queries, attention, output projection."""
        self.project(stream)
        self.attend(stream)
        return self.output(stream)
