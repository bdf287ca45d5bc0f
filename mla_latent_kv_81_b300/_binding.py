"""ctypes binding of libmla.so: argument marshalling only.

Every function here has the name of the C entry point it calls and takes
torch tensors (device memory) instead of raw pointers.  All arithmetic runs
in the library's CUDA kernels; if the library is missing this module raises
at import time rather than falling back to anything else.
"""
from __future__ import annotations

import ctypes
import math
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmla.so")

MLA_F32, MLA_BF16 = 0, 1
STATUS = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED", 3: "MLA_ERR_CUDA",
          4: "MLA_ERR_TIMEOUT", 5: "MLA_ERR_DEVICE_INDEX", 6: "MLA_ERR_WORKSPACE"}


class MlaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {STATUS.get(code, code)}")
        self.code = code


class mla_config(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int), ("n_heads", ctypes.c_int), ("qk_nope", ctypes.c_int),
                ("d_rope", ctypes.c_int), ("v_head", ctypes.c_int), ("d_c", ctypes.c_int),
                ("block_size", ctypes.c_int), ("softmax_scale", ctypes.c_float), ("dtype", ctypes.c_int),
                ("cache_fp8", ctypes.c_int), ("rope_per_head", ctypes.c_int)]


class mla_paged_cache(ctypes.Structure):
    _fields_ = [("pool", ctypes.c_void_p), ("num_blocks", ctypes.c_int), ("block_table", ctypes.c_void_p),
                ("max_blocks_per_seq", ctypes.c_int), ("batch", ctypes.c_int)]


class mla_rope_table(ctypes.Structure):
    _fields_ = [("cos_sin", ctypes.c_void_p), ("max_pos", ctypes.c_int)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run `python -m mla_latent_kv_81_b300.build` "
                          "(or __graft_entry__.build()) first")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, Z, VP = ctypes.POINTER, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
    cfgp, cachep, ropep = P(mla_config), P(mla_paged_cache), P(mla_rope_table)
    sig = {
        "mla_cache_bytes_per_token": (Z, [cfgp]),
        "mla_rope_table_create": (I, [cfgp, ctypes.c_float, I, VP, VP]),
        "mla_compress_workspace_bytes": (Z, [cfgp, I]),
        "mla_compress_append": (I, [cfgp, VP, VP, VP, VP, VP, ropep, cachep, I, VP, Z, VP]),
        "mla_absorb_workspace_bytes": (Z, [cfgp, I]),
        "mla_absorb_query": (I, [cfgp, VP, VP, VP, VP, VP, ropep, VP, I, VP, Z, VP]),
        "mla_decode_workspace_bytes": (Z, [cfgp, I, I, I]),
        "mla_decode_attention": (I, [cfgp, VP, cachep, VP, I, I, VP, VP, VP, Z, VP]),
        "mla_output_workspace_bytes": (Z, [cfgp, I]),
        "mla_output_project": (I, [cfgp, VP, VP, VP, VP, I, VP, Z, VP]),
        "mla_get_device_status": (I, [VP, VP, P(ctypes.c_uint32)]),
        "mla_selftest_wait_timeout": (I, [VP, Z, ctypes.c_uint32, VP]),
        "mla_status_string": (ctypes.c_char_p, [I]),
        "mla_kernel_launches": (ctypes.c_uint64, []),
        "mla_compress_append_noalloc": (I, [cfgp, VP, VP, VP, VP, VP, ropep, cachep, I, VP]),
        "mla_project_workspace_bytes": (Z, [cfgp, I]),
        "mla_project_query": (I, [cfgp, VP, VP, VP, VP, ropep, VP, I, VP, Z, VP]),
        "mla_prefill_workspace_bytes": (Z, [cfgp, I]),
        "mla_prefill_attention": (I, [cfgp, VP, cachep, I, I, I, VP, VP, VP, VP, VP, Z, VP]),
        "mla_head_output_workspace_bytes": (Z, [cfgp, I]),
        "mla_head_output_project": (I, [cfgp, VP, VP, VP, I, VP, Z, VP]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    return lib


lib = _load()
EXPORTED = ("mla_cache_bytes_per_token", "mla_rope_table_create", "mla_compress_workspace_bytes",
            "mla_compress_append", "mla_absorb_workspace_bytes", "mla_absorb_query",
            "mla_decode_workspace_bytes", "mla_decode_attention", "mla_output_workspace_bytes",
            "mla_output_project", "mla_get_device_status", "mla_status_string", "mla_kernel_launches",
            "mla_compress_append_noalloc", "mla_selftest_wait_timeout", "mla_project_workspace_bytes",
            "mla_project_query", "mla_prefill_workspace_bytes", "mla_prefill_attention",
            "mla_head_output_workspace_bytes", "mla_head_output_project")


# ------------------------------------------------------------------ marshalling helpers
def make_config(dims, dtype: str, softmax_scale: float = 0.0, cache_fp8: bool = False,
                rope_per_head: bool = False) -> mla_config:
    return mla_config(dims.d_model, dims.n_heads, dims.qk_nope, dims.d_rope, dims.v_head, dims.d_c,
                      dims.block_size, softmax_scale, MLA_BF16 if dtype == "bf16" else MLA_F32, int(cache_fp8),
                      int(rope_per_head))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn: str, code: int):
    if code != 0:
        raise MlaError(fn, code)


def make_cache(pool, block_table, block_size: int) -> mla_paged_cache:
    """pool: [num_blocks, d_c + d_rope, block_size] (element-major blocks); block_table: int32 [batch, max_blocks]."""
    return mla_paged_cache(pool.data_ptr(), pool.shape[0], block_table.data_ptr(), block_table.shape[1],
                           block_table.shape[0])


def make_rope(cos_sin) -> mla_rope_table:
    return mla_rope_table(cos_sin.data_ptr(), cos_sin.shape[0])


def workspace(nbytes: int, device):
    """A caller workspace of at least `nbytes`, zero-filled (its header's status word starts at zero)."""
    import torch
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ entry points (same names as the C ABI)
def mla_cache_bytes_per_token(cfg: mla_config) -> int:
    return int(lib.mla_cache_bytes_per_token(ctypes.byref(cfg)))


def mla_rope_table_create(cfg: mla_config, base: float, max_pos: int, out, stream=None):
    """out: fp32 device tensor [max_pos, d_rope/2, 2]."""
    _check("mla_rope_table_create",
           lib.mla_rope_table_create(ctypes.byref(cfg), base, max_pos, _ptr(out), _stream(stream)))
    return out


def mla_compress_workspace_bytes(cfg, T):
    return int(lib.mla_compress_workspace_bytes(ctypes.byref(cfg), T))


def mla_compress_append(cfg, x, W_DKV, W_KR, seq_idx, pos, rope: mla_rope_table, cache: mla_paged_cache,
                        ws=None, stream=None):
    T = x.shape[0]
    if ws is None:
        ws = workspace(mla_compress_workspace_bytes(cfg, T), x.device)
    _check("mla_compress_append",
           lib.mla_compress_append(ctypes.byref(cfg), _ptr(x), _ptr(W_DKV), _ptr(W_KR), _ptr(seq_idx), _ptr(pos),
                                   ctypes.byref(rope), ctypes.byref(cache), T, _ptr(ws), ws.numel(),
                                   _stream(stream)))


def mla_compress_append_noalloc(cfg, x, W_DKV, W_KR, seq_idx, pos, rope: mla_rope_table, cache: mla_paged_cache,
                                stream=None):
    """mla_compress_append with its scratch in the library's fixed device array (no workspace)."""
    _check("mla_compress_append_noalloc",
           lib.mla_compress_append_noalloc(ctypes.byref(cfg), _ptr(x), _ptr(W_DKV), _ptr(W_KR), _ptr(seq_idx),
                                           _ptr(pos), ctypes.byref(rope), ctypes.byref(cache), x.shape[0],
                                           _stream(stream)))


def mla_absorb_workspace_bytes(cfg, N):
    return int(lib.mla_absorb_workspace_bytes(ctypes.byref(cfg), N))


def mla_absorb_query(cfg, x, W_Q, W_QR, W_UK, q_pos, rope: mla_rope_table, q_out, ws=None, stream=None):
    N = x.shape[0]
    if ws is None:
        ws = workspace(mla_absorb_workspace_bytes(cfg, N), x.device)
    _check("mla_absorb_query",
           lib.mla_absorb_query(ctypes.byref(cfg), _ptr(x), _ptr(W_Q), _ptr(W_QR), _ptr(W_UK), _ptr(q_pos),
                                ctypes.byref(rope), _ptr(q_out), N, _ptr(ws), ws.numel(), _stream(stream)))
    return q_out


def mla_decode_workspace_bytes(cfg, batch, n_q, max_blocks_per_seq):
    return int(lib.mla_decode_workspace_bytes(ctypes.byref(cfg), batch, n_q, max_blocks_per_seq))


def mla_decode_attention(cfg, q, cache: mla_paged_cache, kv_len, batch, n_q, o_lat, lse=None, ws=None,
                         stream=None):
    if ws is None:
        ws = workspace(mla_decode_workspace_bytes(cfg, batch, n_q, cache.max_blocks_per_seq), q.device)
    _check("mla_decode_attention",
           lib.mla_decode_attention(ctypes.byref(cfg), _ptr(q), ctypes.byref(cache), _ptr(kv_len), batch, n_q,
                                    _ptr(o_lat), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)))
    return o_lat


def mla_output_workspace_bytes(cfg, N):
    return int(lib.mla_output_workspace_bytes(ctypes.byref(cfg), N))


def mla_output_project(cfg, o_lat, W_UV, W_O, out, ws=None, stream=None):
    N = o_lat.shape[0]
    if ws is None:
        ws = workspace(mla_output_workspace_bytes(cfg, N), o_lat.device)
    _check("mla_output_project",
           lib.mla_output_project(ctypes.byref(cfg), _ptr(o_lat), _ptr(W_UV), _ptr(W_O), _ptr(out), N, _ptr(ws),
                                  ws.numel(), _stream(stream)))
    return out


def mla_project_workspace_bytes(cfg, N):
    return int(lib.mla_project_workspace_bytes(ctypes.byref(cfg), N))


def mla_project_query(cfg, x, W_Q, W_QR, q_pos, rope: mla_rope_table, q_out, ws=None, stream=None):
    N = x.shape[0]
    if ws is None:
        ws = workspace(mla_project_workspace_bytes(cfg, N), x.device)
    _check("mla_project_query",
           lib.mla_project_query(ctypes.byref(cfg), _ptr(x), _ptr(W_Q), _ptr(W_QR), _ptr(q_pos), ctypes.byref(rope),
                                 _ptr(q_out), N, _ptr(ws), ws.numel(), _stream(stream)))
    return q_out


def mla_prefill_workspace_bytes(cfg, kv_len):
    return int(lib.mla_prefill_workspace_bytes(ctypes.byref(cfg), kv_len))


def mla_prefill_attention(cfg, q, cache: mla_paged_cache, seq, kv_len, W_UK, W_UV, o, lse=None, ws=None,
                          stream=None):
    T = q.shape[0]
    if ws is None:
        ws = workspace(mla_prefill_workspace_bytes(cfg, kv_len), q.device)
    _check("mla_prefill_attention",
           lib.mla_prefill_attention(ctypes.byref(cfg), _ptr(q), ctypes.byref(cache), seq, kv_len, T, _ptr(W_UK),
                                     _ptr(W_UV), _ptr(o), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)))
    return o


def mla_head_output_workspace_bytes(cfg, N):
    return int(lib.mla_head_output_workspace_bytes(ctypes.byref(cfg), N))


def mla_head_output_project(cfg, o, W_O, out, ws=None, stream=None):
    N = o.shape[0]
    if ws is None:
        ws = workspace(mla_head_output_workspace_bytes(cfg, N), o.device)
    _check("mla_head_output_project",
           lib.mla_head_output_project(ctypes.byref(cfg), _ptr(o), _ptr(W_O), _ptr(out), N, _ptr(ws), ws.numel(),
                                       _stream(stream)))
    return out


def mla_get_device_status(ws=None, stream=None):
    """Returns (status_code, flags) of the calls made with workspace `ws` (the library's own word
    when None), and clears it; synchronises the stream."""
    flags = ctypes.c_uint32(0)
    code = lib.mla_get_device_status(_ptr(ws), _stream(stream), ctypes.byref(flags))
    return int(code), int(flags.value)


def mla_selftest_wait_timeout(ws, limit_cycles: int, stream=None):
    """Run the bounded-wait self-check with workspace `ws` (its status word then reports a timeout)."""
    _check("mla_selftest_wait_timeout",
           lib.mla_selftest_wait_timeout(_ptr(ws), ws.numel(), limit_cycles, _stream(stream)))


def mla_kernel_launches() -> int:
    return int(lib.mla_kernel_launches())


def mla_status_string(code: int) -> str:
    return lib.mla_status_string(code).decode()


def default_scale(dims) -> float:
    return 1.0 / math.sqrt(dims.qk_nope + dims.d_rope)
