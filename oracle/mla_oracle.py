"""Float64 CPU oracle for the MLA decode path.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module.  It shares no code with the CUDA
library and never reads the paged cache layout: it works on logical
(per-sequence, per-position) rows.

Sources, cited as [tag section] below:
  [KJ]  "What does Multi-head Latent Attention compress, and how is that
        different from quantizing the cache?" (katajob.com)
  [ZQ]  "How does DeepSeek's Multi-Latent Attention (MLA) compress the KV cache
        below GQA?" (zenaique.com)
  [BB]  "Multi-head Latent Attention (MLA)" (bembew.net)
  [TM]  "Multi-head Latent Attention" knowledge card mla-attention (talentme)
  [SC]  "What Is Multi-head Latent Attention—and How Does It Shrink AI's
        Memory?" (satishkchoudhary.com, transcript)

Readings where the pages are silent or garbled (each repeated in the design doc):
  * weights are stored [out, in]; a projection is W @ x             (c8)
  * one decoupled RoPE key k_R per token, shared by all heads; each
    head has its own rotated query part q_R                          (c1)
  * the content key and the RoPE key are concatenated, so a score is
    the sum of the two dot products                                  (c2)
  * scale = 1/sqrt(qk_nope + d_rope)                                 (c3)
  * RoPE rotates interleaved pairs (2i, 2i+1), theta_i = base^(-2i/d_r) (c4)
  * query j of a sequence sees vis_j = kv_len - (n_q - 1 - j) tokens (c5)
  * no query compression, no norms, no biases                        (c6)
  * an empty visible set gives a zero output                         (c10)

Every function computes in float64 on float64 copies of its inputs.
Parity: every function below is pinned by a test in tests/test_oracle.py
(brute force, invariants, special cases, closed forms); see the table in
the design doc.  The only unpinned claim (model quality on real benchmarks) is
not computed here.
"""
from __future__ import annotations

import numpy as np

f64 = np.float64


def _a(x) -> np.ndarray:
    return np.asarray(x, dtype=f64)


# ------------------------------------------------------------------ storage rounding
def round_bf16(x) -> np.ndarray:
    """Nearest bfloat16 value of each element (ties to even), returned as float64.

    bfloat16 keeps 8 significant bits: for |x| in [2^e, 2^(e+1)) the spacing is
    2^(e-7).  Used only where the bf16 pipeline stores a value (reading c9:
    cached c and k_R, the absorbed query, the latent output), to give each stage
    check the inputs the method specifies.
    """
    x = _a(x)
    out = np.zeros_like(x)
    nz = (x != 0) & np.isfinite(x)
    ax = np.abs(x[nz])
    e = np.floor(np.log2(ax))
    spacing = np.power(2.0, e - 7)
    q = ax / spacing                       # in [128, 256)
    r = np.floor(q)
    frac = q - r
    r = np.where(frac > 0.5, r + 1, np.where(frac < 0.5, r, r + (r % 2)))
    out[nz] = np.sign(x[nz]) * r * spacing
    out[~np.isfinite(x)] = x[~np.isfinite(x)]
    return out


# ------------------------------------------------------------------ RoPE
def rope_angles(pos, d_rope: int, base: float = 10000.0) -> np.ndarray:
    """phi[p, i] = pos_p * base^(-2i/d_rope), i < d_rope/2.

    [BB §2 Decoupling RoPE from Compression]: RoPE injects position by a
    position-dependent rotation; the frequencies follow reading c4.
    """
    pos = _a(pos).reshape(-1)
    i = np.arange(d_rope // 2, dtype=f64)
    theta = np.power(f64(base), -2.0 * i / d_rope)
    return pos[:, None] * theta[None, :]


def apply_rope(v, pos, base: float = 10000.0) -> np.ndarray:
    """Rotate each interleaved pair (v[2i], v[2i+1]) of the last axis by phi_i(pos).

    v: [..., d_rope]; pos broadcast against v's leading axes.
    [a, b] -> [a cos phi - b sin phi, a sin phi + b cos phi].
    """
    v = _a(v)
    d_rope = v.shape[-1]
    lead = v.shape[:-1]
    pos = np.broadcast_to(_a(pos), lead)
    phi = rope_angles(pos.reshape(-1), d_rope, base).reshape(*lead, d_rope // 2)
    a, b = v[..., 0::2], v[..., 1::2]
    cos, sin = np.cos(phi), np.sin(phi)
    out = np.empty_like(v)
    out[..., 0::2] = a * cos - b * sin
    out[..., 1::2] = a * sin + b * cos
    return out


# ------------------------------------------------------------------ projections
def compress(x, W_DKV, W_KR, pos, base: float = 10000.0):
    """Latent and decoupled RoPE key of each token: c_t = W_DKV x_t, k_R,t = RoPE(W_KR x_t, pos_t).

    [KJ §The mechanism] down-projection into one latent per token, the only
    thing retained; [BB §1 eq.] c_KV^t; [BB Implementation Logic] steps 1, 3, 4
    (latent = h W_down, K_rope = h W_rope, then RoPE); [TM Core Definition] k_t^R.
    Returns (c [T, d_c], k_R [T, d_rope]).
    """
    x = _a(x)
    c = x @ _a(W_DKV).T
    k_r = apply_rope(x @ _a(W_KR).T, _a(pos), base)
    return c, k_r


def compress_per_head_rope(x, W_DKV, W_KR, pos, n_heads: int, base: float = 10000.0):
    """The per-head positional-key variant ([ZQ] "a small per-head RoPE-carrying key"; the alternative
    to reading c1): k_R^h,t = RoPE(W_KR^h x_t, pos_t) for every head, W_KR stored [n_heads * d_rope]
    [d_model] (head h's rows h*d_rope .. h*d_rope + d_rope - 1), the rotation frequencies restarting in
    every head's key.  Returns (c [T, d_c], k_R [T, n_heads, d_rope])."""
    x = _a(x)
    c = x @ _a(W_DKV).T
    y = x @ _a(W_KR).T
    y = y.reshape(x.shape[0], n_heads, -1)
    k_r = apply_rope(y, _a(pos)[:, None], base)
    return c, k_r


def project_query(x, W_Q, W_QR, q_pos, n_heads: int, base: float = 10000.0):
    """Per-head content query q_nope^h = W_Q^h x and rotated query q_R^h = RoPE(W_QR^h x, q_pos).

    [KJ §The mechanism] query projection; [ZQ decoupled RoPE question] the
    positional part is kept out of the absorbable path (reading c1, c6).
    Returns (q_nope [N, H, qk_nope], q_rope [N, H, d_rope]).
    """
    x = _a(x)
    N = x.shape[0]
    q_nope = (x @ _a(W_Q).T).reshape(N, n_heads, -1)
    q_rope_raw = (x @ _a(W_QR).T).reshape(N, n_heads, -1)
    q_rope = apply_rope(q_rope_raw, _a(q_pos).reshape(N, 1), base)
    return q_nope, q_rope


def reconstruct_kv(c, W_UK, W_UV, h: int):
    """Explicit per-head key content and value: k_t^h = W_UK^h c_t, v_t^h = W_UV^h c_t.

    [KJ solid answer] up-projections expand the latent into every head's keys
    and values; [BB §1 eq.] K^t = W c^t, V^t = W c^t (the page's matrix names
    are garbled; reading c7 treats both as up-projections).
    """
    c = _a(c)
    return c @ _a(W_UK)[h].T, c @ _a(W_UV)[h].T


def softmax_scale(qk_nope: int, d_rope: int) -> float:
    """Reading c3: 1/sqrt of the full explicit key width."""
    return 1.0 / np.sqrt(qk_nope + d_rope)


def visible(kv_len: int, n_q: int, j: int) -> int:
    """Reading c5: query j of n_q sees the first kv_len - (n_q - 1 - j) cached tokens."""
    return max(0, int(kv_len) - (n_q - 1 - j))


def _softmax_weights(s: np.ndarray):
    """Max-subtracted softmax over the last axis, float64; also returns log-sum-exp."""
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    z = np.sum(e, axis=-1, keepdims=True)
    return e / z, (m + np.log(z))[..., 0]


# ------------------------------------------------------------------ explicit attention
def attend_explicit(q_nope, q_rope, c, k_r, W_UK, W_UV, kv_len: int, scale: float | None = None):
    """Standard multi-head softmax attention for one sequence, with K and V rebuilt per head.

    This is the plain definition the absorbed decode path must reproduce:
      k_t^h = [W_UK^h c_t || k_R,t],  v_t^h = W_UV^h c_t,
      s_t^h = scale * (q_nope^h . W_UK^h c_t + q_R^h . k_R,t),  t < vis_j,
      o^h   = sum_t softmax(s^h)_t v_t^h.
    [KJ §The mechanism, solid answer]; [BB §1 eq., §2, Implementation Logic
    step 5: content and positional key combined, reading c2]; [SC] every prior
    token keeps an entry (no token selection).
    q_nope [n_q, H, qk_nope], q_rope [n_q, H, d_rope], c [L, d_c], k_r [L, d_rope], or [L, H, d_rope]
    with a positional key per head (head h scores q_R^h against its own k_R^h).
    Returns o [n_q, H, v_head].
    """
    q_nope, q_rope, c, k_r = _a(q_nope), _a(q_rope), _a(c), _a(k_r)
    n_q, H, _ = q_nope.shape
    if scale is None:
        scale = softmax_scale(q_nope.shape[-1], q_rope.shape[-1])
    v_head = _a(W_UV).shape[1]
    out = np.zeros((n_q, H, v_head), dtype=f64)
    for h in range(H):
        K_h, V_h = reconstruct_kv(c, W_UK, W_UV, h)       # [L, qk_nope], [L, v_head]
        for j in range(n_q):
            vis = visible(kv_len, n_q, j)
            if vis == 0:
                continue                                   # reading c10
            kr = k_r[:vis, h] if k_r.ndim == 3 else k_r[:vis]
            s = scale * (K_h[:vis] @ q_nope[j, h] + kr @ q_rope[j, h])
            p, _ = _softmax_weights(s)
            out[j, h] = p @ V_h[:vis]
    return out


def attend_explicit_at(q_nope, q_rope, pos, c, k_r, W_UK, W_UV, scale: float, store=None):
    """Explicit attention for queries at given positions of one sequence: query j
    sees the tokens at positions 0..pos[j] (a prompt at prefill, every prompt
    token a query: [TM point 4], keys and values recomputed from the latent;
    visibility is reading c5 with the query's own row already cached).

    The same definition as attend_explicit -- K and V rebuilt per head from c,
    score = scale (q_nope . k + q_R . k_R), softmax, weighted sum of V -- with
    each head's K and V rebuilt once for all the queries.
    q_nope [n, H, qk_nope], q_rope [n, H, d_rope], pos int [n], c [L, d_c],
    k_r [L, d_rope] with L > max(pos).
    store: applied to each head's rebuilt K and V before use (a bf16 pipeline
    stores them in bf16: pass round_bf16, reading c20); default keeps them exact.
    Returns o [n, H, v_head] and lse [n, H] (natural log of the softmax
    normaliser of the scaled scores).
    """
    q_nope, q_rope, c, k_r = _a(q_nope), _a(q_rope), _a(c), _a(k_r)
    pos = np.asarray(pos, dtype=np.int64)
    n, H, _ = q_nope.shape
    v_head = _a(W_UV).shape[1]
    top = int(pos.max()) + 1
    o = np.zeros((n, H, v_head), dtype=f64)
    lse = np.zeros((n, H), dtype=f64)
    for h in range(H):
        K_h, V_h = reconstruct_kv(c[:top], W_UK, W_UV, h)
        if store is not None:
            K_h, V_h = store(K_h), store(V_h)
        for j in range(n):
            vis = int(pos[j]) + 1
            kr = k_r[:vis, h] if k_r.ndim == 3 else k_r[:vis]
            s = scale * (K_h[:vis] @ q_nope[j, h] + kr @ q_rope[j, h])
            p, lse[j, h] = _softmax_weights(s)
            o[j, h] = p @ V_h[:vis]
    return o, lse


def output_project(o, W_O):
    """out = W_O concat_h(o^h).  [KJ §Why it is not just extra work] output projection."""
    o = _a(o)
    N = o.shape[0]
    return o.reshape(N, -1) @ _a(W_O).T


# ------------------------------------------------------------------ absorbed (latent) form
def absorb_query(q_nope, W_UK):
    """q_abs^h = W_UK^h^T q_nope^h, so that q_abs^h . c_t = q_nope^h . (W_UK^h c_t).

    [KJ §Why it is not just extra work]: the key up-projection is folded into
    the query; [ZQ concept explanation]: reconstruction fused into the
    attention matmuls.  q_nope [N, H, qk_nope] -> [N, H, d_c].
    """
    return np.einsum("nhi,hic->nhc", _a(q_nope), _a(W_UK))


def attend_latent(q_abs, q_rope, c, k_r, kv_len: int, scale: float):
    """Attention scored and accumulated in latent space for one sequence.

      s_t^h = scale * (q_abs^h . c_t + q_R^h . k_R,t),  t < vis_j
      o_lat^h = sum_t softmax(s^h)_t c_t,  lse^h = log sum_t exp(s_t^h)
    [KJ §Why it is not just extra work]: after folding, attention runs in
    the latent space directly and per-head K, V are never formed.
    q_abs [n_q, H, d_c], q_rope [n_q, H, d_rope] -> (o_lat [n_q, H, d_c], lse [n_q, H]).
    An empty visible set gives o_lat = 0 and lse = -inf (reading c10).
    """
    q_abs, q_rope, c, k_r = _a(q_abs), _a(q_rope), _a(c), _a(k_r)
    n_q, H, d_c = q_abs.shape
    o_lat = np.zeros((n_q, H, d_c), dtype=f64)
    lse = np.full((n_q, H), -np.inf, dtype=f64)
    for j in range(n_q):
        vis = visible(kv_len, n_q, j)
        if vis == 0:
            continue
        s = scale * (q_abs[j] @ c[:vis].T + q_rope[j] @ k_r[:vis].T)   # [H, vis]
        p, lse[j] = _softmax_weights(s)
        o_lat[j] = p @ c[:vis]
    return o_lat, lse


def up_project_values(o_lat, W_UV):
    """o^h = W_UV^h o_lat^h: the value up-projection applied after the weighted sum.

    [KJ §Why it is not just extra work]: the value up-projection is folded
    into the output side.  o_lat [N, H, d_c] -> [N, H, v_head].
    """
    return np.einsum("hvc,nhc->nhv", _a(W_UV), _a(o_lat))


def merge_partials(o_parts, lse_parts):
    """Combine attention results over disjoint token ranges of one query.

    o = sum_s exp(lse_s - lse) o_s, lse = log sum_s exp(lse_s).  This is the
    exact identity softmax over a union = weighted softmaxes over the parts.
    o_parts [S, ..., d], lse_parts [S, ...].
    """
    o_parts, lse_parts = _a(o_parts), _a(lse_parts)
    m = np.max(lse_parts, axis=0)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    w = np.exp(lse_parts - m_safe)
    z = np.sum(w, axis=0)
    lse = np.where(z > 0, m_safe + np.log(np.where(z > 0, z, 1.0)), -np.inf)
    o = np.sum(w[..., None] * o_parts, axis=0) / np.where(z > 0, z, 1.0)[..., None]
    return o, lse


# ------------------------------------------------------------------ whole layer
def decode_layer_explicit(x_q, q_pos, caches, W, dims, n_q: int, kv_len):
    """End-to-end explicit form for a batch: query projection, per-head MHA over
    rebuilt K/V, output projection.  caches[b] = (c [L_b, d_c], k_r [L_b, d_rope])."""
    q_nope, q_rope = project_query(x_q, W["W_Q"], W["W_QR"], q_pos, dims.n_heads, dims.rope_base)
    B = len(caches)
    o = np.zeros((B * n_q, dims.n_heads, dims.v_head), dtype=f64)
    scale = softmax_scale(dims.qk_nope, dims.d_rope)
    for b in range(B):
        c, k_r = caches[b]
        sl = slice(b * n_q, (b + 1) * n_q)
        o[sl] = attend_explicit(q_nope[sl], q_rope[sl], c, k_r, W["W_UK"], W["W_UV"], int(kv_len[b]), scale)
    return output_project(o, W["W_O"])


def decode_layer_absorbed(x_q, q_pos, caches, W, dims, n_q: int, kv_len):
    """The same layer computed the absorbed way (used only as an invariant check)."""
    q_nope, q_rope = project_query(x_q, W["W_Q"], W["W_QR"], q_pos, dims.n_heads, dims.rope_base)
    q_abs = absorb_query(q_nope, W["W_UK"])
    B = len(caches)
    o_lat = np.zeros((B * n_q, dims.n_heads, dims.d_c), dtype=f64)
    scale = softmax_scale(dims.qk_nope, dims.d_rope)
    for b in range(B):
        c, k_r = caches[b]
        sl = slice(b * n_q, (b + 1) * n_q)
        o_lat[sl], _ = attend_latent(q_abs[sl], q_rope[sl], c, k_r, int(kv_len[b]), scale)
    return output_project(up_project_values(o_lat, W["W_UV"]), W["W_O"])


# ------------------------------------------------------------------ reduced-precision latent cache
# [KJ "Compression as architecture versus compression as post-processing"]: a latent representation
# can itself be stored in a reduced-precision format.  Reading c21 (the pages name no format): FP8 E4M3
# codes (4 exponent bits, bias 7, 3 mantissa bits, subnormals below 2^-6, largest finite 448) of
# c_t / s_t with one power-of-two scale s_t per token, the smallest with max|c_t| / s_t <= 448; the
# positional key is kept in bf16, stored divided by the same s_t (exact for a power of two).
E4M3_MAX = 448.0


def round_e4m3(x) -> np.ndarray:
    """Nearest FP8 E4M3 value of each element (ties to even), for |x| <= 448.

    Normal values 2^e (1 + m/8), e >= -6, have spacing 2^(e-3); below 2^-6 the spacing is 2^-9."""
    x = _a(x)
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    q = 2.0 ** (np.maximum(e, -6.0) - 3.0)
    return np.sign(x) * np.round(a / q) * q          # numpy rounds halves to even


def e4m3_value(code) -> np.ndarray:
    """The value of each FP8 E4M3 bit pattern (uint8): sign, 4-bit exponent (bias 7), 3-bit mantissa;
    exponent 0 is subnormal (m/8 * 2^-6); pattern 0x7F / 0xFF (NaN) gives nan."""
    c = np.asarray(code, dtype=np.int64)
    sgn = np.where(c & 0x80, -1.0, 1.0)
    e, m = (c >> 3) & 0xF, c & 0x7
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))
    return np.where((c & 0x7F) == 0x7F, np.nan, sgn * val)


def fp8_token_scale(c) -> np.ndarray:
    """Reading c21: per token (last axis) the smallest power of two s with max|c| / s <= 448; 1 when
    the row is all zeros."""
    m = np.max(np.abs(_a(c)), axis=-1)
    k = np.ceil(np.log2(np.where(m > 0, m, E4M3_MAX) / E4M3_MAX))
    return 2.0 ** k


def quantize_latent_fp8(c, k_r):
    """A cache row in the reduced-precision format (reading c21): returns (codes as values, s, k_R / s
    rounded to bf16).  The stored latent is codes * s, the stored positional key (k_R / s) * s."""
    c, k_r = _a(c), _a(k_r)
    s = fp8_token_scale(c)
    return round_e4m3(c / s[..., None]), s, round_bf16(k_r / s[..., None])


def dequantize_latent_fp8(codes, s, k_r_scaled):
    """Latent and positional key a reduced-precision cache row stands for: (codes * s, k_R' * s)."""
    s = _a(s)[..., None]
    return _a(codes) * s, _a(k_r_scaled) * s


# ------------------------------------------------------------------ cache-size closed forms
def kv_cache_elems_per_token(n_kv_heads: int, d_head: int, n_layers: int = 1) -> int:
    """Head-sharing / MHA cache: keys and values per KV head, 2 * H_kv * d per layer.

    [ZQ What MLA caches versus what MHA and GQA cache]; [TM Key Problems
    Solved] 2Hd per token; [SC] the 32 x 8 x 128 x 2 worked example.
    """
    return 2 * n_kv_heads * d_head * n_layers


def mla_cache_elems_per_token(d_c: int, d_rope: int, n_layers: int = 1) -> int:
    """MLA cache: the latent plus the decoupled RoPE key, d_c + d_rope per layer.

    [TM Key Problems Solved] per-token cache d_c; [SC] compact latent plus
    the smaller positional component; [ZQ] the latent is the only content
    written to the cache.
    """
    return (d_c + d_rope) * n_layers


def cache_bytes(n_tokens: int, elems_per_token: int, bytes_per_elem: int) -> int:
    return int(n_tokens) * int(elems_per_token) * int(bytes_per_elem)
