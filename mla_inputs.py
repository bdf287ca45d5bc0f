"""Seeded synthetic inputs shared by the tests, the benchmark and the CPU oracle checks.

This module only *draws* numbers and lays them out (shapes, bf16 rounding of
the drawn values, paged block tables, NaN sentinels).  It contains none of the
attention arithmetic: nothing here projects, rotates, scores or normalises.

Workloads are shaped like the DeepSeek-V2 layer the pages describe
("How does DeepSeek's Multi-Latent Attention (MLA) compress the KV cache below
GQA?", zenaique, section "What MLA caches versus what MHA and GQA cache":
latent width on the order of 512; "Multi-head Latent Attention" card,
talentme, "Core Definition": d_c = 512), plus the tiny layer whose sizes
match the numpy snippet of "What does Multi-head Latent Attention compress,
and how is that different from quantizing the cache?" (katajob, "code").

Recipe (all draws from ``numpy.random.default_rng``, PCG64):
  * main stream, seeded with the workload seed, in this order:
      W_DKV, W_KR, W_Q, W_QR, W_UK, W_UV, W_O   ~ N(0, 1/fan_in)
      cached lengths (uniform integers, inclusive bounds)
      x_ctx ~ N(0,1)       (only for workloads whose cache is built by append)
      x_q   ~ N(0,1)       (hidden states of the new / query tokens)
      block permutation
  * latent rows for directly filled caches come from one sub-stream per
    sequence (seed sequence [seed, 1000 + b]) so a single sequence can be
    regenerated without drawing the whole cache.
  * everything is drawn in float32; bf16 workloads round each value to bf16
    (round to nearest even) before use, so the oracle sees exactly the values
    the GPU stores.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 64
SPARE_BLOCKS = 8


@dataclass(frozen=True)
class Dims:
    d_model: int
    n_heads: int
    qk_nope: int
    d_rope: int
    v_head: int
    d_c: int
    block_size: int = BLOCK_SIZE
    rope_base: float = 10000.0

    @property
    def row(self) -> int:
        """Elements in one cached row: latent then positional key."""
        return self.d_c + self.d_rope


TINY = Dims(d_model=512, n_heads=8, qk_nope=64, d_rope=16, v_head=64, d_c=64)
DSV2 = Dims(d_model=5120, n_heads=128, qk_nope=128, d_rope=64, v_head=128, d_c=512)


@dataclass(frozen=True)
class Workload:
    name: str
    dims: Dims
    dtype: str            # "f32" or "bf16"
    batch: int
    len_lo: int           # cached tokens per sequence before the step (inclusive bounds)
    len_hi: int
    n_q: int              # query tokens per sequence
    n_append: int         # query tokens appended to the cache before attention (0 or n_q)
    seed: int
    fill: str             # "append": cache built with compress_append; "direct": latent rows drawn
    note: str = ""
    cache_fp8: bool = False   # reduced-precision cache (FP8 E4M3 latent codes, per-token scale)

    @property
    def fixed_len(self) -> bool:
        return self.len_lo == self.len_hi


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_f32_b1_ctx10", TINY, "f32", 1, 10, 10, 1, 0, 0, "append",
                 "10 cached tokens built by append at positions 0..9, one query at position 10"),
        Workload("dsv2_b16_ctx4096", DSV2, "bf16", 16, 4096, 4096, 1, 0, 2, "append",
                 "cache built by appending 65,536 tokens"),
        Workload("dsv2_b64_ctx1k_8k", DSV2, "bf16", 64, 1024, 8192, 1, 0, 3, "direct",
                 "ragged lengths"),
        Workload("dsv2_b64_ctx8192", DSV2, "bf16", 64, 8191, 8191, 1, 1, 33, "direct",
                 "decode step: 8191 cached + the new token appended = 8192 attended per sequence"),
        Workload("dsv2_b4_ctx65536", DSV2, "bf16", 4, 65536, 65536, 1, 0, 4, "direct",
                 "long context, split-KV"),
        Workload("dsv2_b128_ctx4k_32k_nq2", DSV2, "bf16", 128, 4096, 32768, 2, 2, 5, "direct",
                 "two new tokens appended, causal between them"),
        Workload("dsv2_b64_ctx8192_fp8", DSV2, "bf16", 64, 8191, 8191, 1, 1, 34, "direct",
                 "the decode step over a reduced-precision cache (drawn codes, scales and keys; the new "
                 "token quantised by the append)", cache_fp8=True),
        Workload("dsv2_b16_ctx4096_fp8", DSV2, "bf16", 16, 4096, 4096, 1, 0, 35, "append",
                 "reduced-precision cache built by appending 65,536 tokens", cache_fp8=True),
    ]
}


# ---------------------------------------------------------------- bf16 helpers
def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    bits = a.view(np.uint32).astype(np.uint64)
    bias = ((bits >> 16) & 1) + 0x7FFF
    out = ((bits + bias) & 0xFFFF0000).astype(np.uint32)
    return out.view(np.float32).reshape(a.shape)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of float32 values that are already bf16-exact."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def storage(a: np.ndarray, dtype: str) -> np.ndarray:
    return round_to_bf16(a) if dtype == "bf16" else np.asarray(a, dtype=np.float32)


# ---------------------------------------------------------------- draws
def main_rng(w: Workload) -> np.random.Generator:
    return np.random.default_rng(w.seed)


def _normal(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    out = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    return out


def draw_weights(dims: Dims, dtype: str, rng: np.random.Generator) -> dict:
    """Weights stored [out_features, in_features] (per-head up-projections [H, out, d_c])."""
    H = dims.n_heads
    spec = [
        ("W_DKV", (dims.d_c, dims.d_model), dims.d_model),
        ("W_KR", (dims.d_rope, dims.d_model), dims.d_model),
        ("W_Q", (H * dims.qk_nope, dims.d_model), dims.d_model),
        ("W_QR", (H * dims.d_rope, dims.d_model), dims.d_model),
        ("W_UK", (H, dims.qk_nope, dims.d_c), dims.d_c),
        ("W_UV", (H, dims.v_head, dims.d_c), dims.d_c),
        ("W_O", (dims.d_model, H * dims.v_head), H * dims.v_head),
    ]
    return {name: storage(_normal(rng, shape, 1.0 / np.sqrt(fan_in)), dtype) for name, shape, fan_in in spec}


def draw_lengths(w: Workload, rng: np.random.Generator) -> np.ndarray:
    if w.fixed_len:
        return np.full(w.batch, w.len_lo, dtype=np.int64)
    return rng.integers(w.len_lo, w.len_hi, size=w.batch, endpoint=True).astype(np.int64)


def draw_hidden(rng: np.random.Generator, n: int, d_model: int, dtype: str) -> np.ndarray:
    return storage(_normal(rng, (n, d_model), 1.0), dtype)


def draw_latent_rows(w: Workload, b: int, n_rows: int) -> np.ndarray:
    """Directly drawn cache rows [n_rows, d_c + d_rope] for sequence b (its own sub-stream)."""
    rng = np.random.default_rng([w.seed, 1000 + b])
    return storage(_normal(rng, (n_rows, w.dims.row), 1.0), w.dtype)


def draw_fp8_rows(w: Workload, b: int, n_rows: int):
    """Directly drawn rows of a reduced-precision cache for sequence b (its own sub-stream): latent
    codes as FP8 E4M3 bit patterns (random sign, exponent field 6..14, mantissa 0..7: magnitudes
    0.5..480 before the scale), the per-token scale exponent k (uniform in -9..-7; scale 2^k) and the
    stored positional key k_R / 2^k (bf16 values of a Gaussian of standard deviation 2^-k, so that the
    key itself has unit spread).  Returns (codes uint8 [n, d_c], k int [n], kr_scaled float32 [n, d_rope])."""
    d = w.dims
    rng = np.random.default_rng([w.seed, 2000 + b])
    sign = rng.integers(0, 2, size=(n_rows, d.d_c)) << 7
    expo = rng.integers(6, 15, size=(n_rows, d.d_c)) << 3
    mant = rng.integers(0, 8, size=(n_rows, d.d_c))
    codes = (sign | expo | mant).astype(np.uint8)
    k = rng.integers(-9, -6, size=n_rows)
    kr = _normal(rng, (n_rows, d.d_rope), 1.0) * (2.0 ** -k)[:, None].astype(np.float32)
    return codes, k.astype(np.int32), round_to_bf16(kr)


def draw_block_table(capacity: np.ndarray, block_size: int, rng: np.random.Generator,
                     spare: int = SPARE_BLOCKS):
    """Shuffled physical blocks for each sequence's logical blocks.

    Returns (block_table [B, max_blocks] int32 with -1 in unused entries,
    num_blocks including ``spare`` never-referenced blocks).
    """
    nblk = [(int(c) + block_size - 1) // block_size for c in capacity]
    total = int(sum(nblk))
    perm = rng.permutation(total).astype(np.int32)
    max_blocks = max(nblk) if nblk else 0
    table = np.full((len(capacity), max(max_blocks, 1)), -1, dtype=np.int32)
    k = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[k:k + n]
        k += n
    return table, total + spare


@dataclass
class Problem:
    """Everything one workload step needs, on the host, in logical (unpaged) order."""
    w: Workload
    weights: dict
    lens: np.ndarray            # cached tokens before the step
    kv_len: np.ndarray          # tokens in the cache during attention
    x_ctx: np.ndarray | None    # [sum(lens), d_model] for append-built caches
    x_q: np.ndarray             # [B * n_q, d_model]
    q_pos: np.ndarray           # [B * n_q] int32
    block_table: np.ndarray
    num_blocks: int
    extra: dict = field(default_factory=dict)

    @property
    def dims(self) -> Dims:
        return self.w.dims


def make_problem(w: Workload, with_weights: bool = True, lens=None) -> Problem:
    """Draw one workload in the documented order (weights are always drawn so
    that the stream stays aligned; ``with_weights=False`` only drops them).
    ``lens`` replaces the drawn cached lengths (test cases with chosen raggedness)."""
    rng = main_rng(w)
    d = w.dims
    weights = draw_weights(d, w.dtype, rng)
    lens_drawn = draw_lengths(w, rng)
    lens = lens_drawn if lens is None else np.asarray(lens, dtype=np.int64)
    assert len(lens) == w.batch
    x_ctx = draw_hidden(rng, int(lens.sum()), d.d_model, w.dtype) if w.fill == "append" else None
    x_q = draw_hidden(rng, w.batch * w.n_q, d.d_model, w.dtype)
    kv_len = lens + w.n_append
    table, num_blocks = draw_block_table(kv_len, d.block_size, rng)
    q_pos = (lens[:, None] + np.arange(w.n_q)[None, :]).reshape(-1).astype(np.int32)
    if not with_weights:
        weights = {}
    return Problem(w, weights, lens, kv_len, x_ctx, x_q, q_pos, table, num_blocks)


def paged_slots(block_table: np.ndarray, b: int, positions: np.ndarray, block_size: int) -> np.ndarray:
    """Physical row index (block * block_size + offset) of logical positions of sequence b."""
    positions = np.asarray(positions, dtype=np.int64)
    return block_table[b, positions // block_size].astype(np.int64) * block_size + positions % block_size


# ---------------------------------------------------------------- prefill (explicit form)
@dataclass(frozen=True)
class PrefillCase:
    """A prompt of `prompt` tokens (positions 0..prompt-1) held by sequence `seq` of a small batch whose
    other sequences hold `others` tokens each: their blocks interleave with the prompt's in the shuffled
    block table and stay unwritten (NaN sentinels).  The last `queries` prompt tokens are the queries.
    fill "direct": cache rows and queries [q_nope || q_R] are drawn directly (the attention stage alone);
    fill "append": the prompt's hidden states are drawn and everything else is computed from them."""
    name: str
    dims: Dims
    dtype: str
    prompt: int
    queries: int
    seed: int
    fill: str = "direct"
    others: tuple = (100, 37)
    seq: int = 1
    note: str = ""
    cache_fp8: bool = False   # reduced-precision cache (fill "append" only)
    rope_per_head: bool = False   # one positional key per head (row d_c + H d_rope; W_KR [H d_rope][d_model])


PREFILL_CASES = {
    c.name: c
    for c in [
        PrefillCase("prefill_dsv2_L300_T300", DSV2, "bf16", 300, 300, 40, note="whole prompt, ragged tiles"),
        PrefillCase("prefill_dsv2_L700_T200", DSV2, "bf16", 700, 200, 41,
                    note="the last 200 tokens of 700: query tiles straddle key tiles"),
        PrefillCase("prefill_dsv2_L300_T1", DSV2, "bf16", 300, 1, 42, note="one query"),
        PrefillCase("prefill_dsv2_L64_T64", DSV2, "bf16", 64, 64, 43, note="one cache block"),
        PrefillCase("prefill_dsv2_L1_T1", DSV2, "bf16", 1, 1, 44, others=(5,), seq=0, note="a single token"),
        PrefillCase("prefill_dsv2_L333_T333_x", DSV2, "bf16", 333, 333, 45, fill="append",
                    note="from hidden states: append, query projection, attention, output projection"),
        PrefillCase("prefill_dsv2_L4096_T4096", DSV2, "bf16", 4096, 4096, 46,
                    note="a 4096-token prompt (benchmark size)"),
        PrefillCase("prefill_dsv2_L8192_T8192", DSV2, "bf16", 8192, 8192, 47, note="an 8192-token prompt"),
        PrefillCase("prefill_dsv2_L333_T200_x_fp8", DSV2, "bf16", 333, 200, 48, fill="append", cache_fp8=True,
                    note="from hidden states over a reduced-precision cache"),
        PrefillCase("prefill_dsv2_L300_T300_rh", DSV2, "bf16", 300, 300, 49, rope_per_head=True,
                    note="per-head positional keys, drawn rows"),
        PrefillCase("prefill_dsv2_L333_T333_x_rh", DSV2, "bf16", 333, 333, 50, fill="append", rope_per_head=True,
                    note="per-head positional keys, from hidden states"),
        PrefillCase("prefill_dsv2_L4096_T4096_rh", DSV2, "bf16", 4096, 4096, 51, rope_per_head=True,
                    note="per-head positional keys, 4096-token prompt"),
    ]
}


@dataclass
class PrefillProblem:
    case: PrefillCase
    weights: dict
    x: np.ndarray | None        # [prompt, d_model] hidden states (fill "append")
    rows: np.ndarray | None     # [prompt, d_c + d_rope] cache rows (fill "direct")
    q: np.ndarray | None        # [queries, H, qk_nope + d_rope] queries (fill "direct")
    lens: np.ndarray            # cached tokens of every sequence of the batch
    block_table: np.ndarray
    num_blocks: int

    @property
    def dims(self) -> Dims:
        return self.case.dims

    @property
    def q_pos(self) -> np.ndarray:
        return np.arange(self.case.prompt - self.case.queries, self.case.prompt, dtype=np.int32)


def make_prefill(c: PrefillCase, sharp: float = 1.0) -> PrefillProblem:
    """Draw a prefill case: main stream seeded with c.seed; weights, then the hidden states (append) or
    the cache rows and queries (direct, queries scaled by `sharp` before rounding), then the block
    permutation."""
    rng = np.random.default_rng(c.seed)
    d = c.dims
    weights = draw_weights(d, c.dtype, rng)
    row = d.d_c + (d.n_heads if c.rope_per_head else 1) * d.d_rope
    if c.rope_per_head:
        # one positional-key projection per head, drawn after the shared-key weights
        weights["W_KR"] = storage(_normal(rng, (d.n_heads * d.d_rope, d.d_model), 1.0 / np.sqrt(d.d_model)), c.dtype)
    x = rows = q = None
    if c.fill == "append":
        x = draw_hidden(rng, c.prompt, d.d_model, c.dtype)
    else:
        rows = storage(_normal(rng, (c.prompt, row), 1.0), c.dtype)
        qq = _normal(rng, (c.queries, d.n_heads, d.qk_nope + d.d_rope), 1.0)
        if sharp != 1.0:
            qq *= np.float32(sharp)
        q = storage(qq, c.dtype)
    lens = list(c.others)
    lens.insert(c.seq, c.prompt)
    lens = np.asarray(lens, dtype=np.int64)
    table, num_blocks = draw_block_table(lens, d.block_size, rng)
    return PrefillProblem(c, weights, x, rows, q, lens, table, num_blocks)


# ---------------------------------------------------------------- stage inputs
def draw_stage_query(dims: Dims, dtype: str, n: int, seed: int, sharp: float = 1.0) -> np.ndarray:
    """Absorbed query rows [n, H, d_c + d_rope] drawn directly, for testing attention alone.

    The latent part has std 0.5 and the positional part std 1, the spread of
    W_UK^T W_Q x and W_QR x with the weight scalings above; ``sharp``
    multiplies both (sharper softmax).
    """
    rng = np.random.default_rng([seed, 7])
    q = rng.standard_normal((n, dims.n_heads, dims.row), dtype=np.float32)
    q[..., :dims.d_c] *= np.float32(0.5)
    if sharp != 1.0:
        q *= np.float32(sharp)
    return storage(q, dtype)


def draw_stage_latent_out(dims: Dims, dtype: str, n: int, seed: int) -> np.ndarray:
    """Latent attention outputs [n, H, d_c] drawn directly, for testing the output projection alone."""
    rng = np.random.default_rng([seed, 8])
    return storage(rng.standard_normal((n, dims.n_heads, dims.d_c), dtype=np.float32), dtype)
