"""Shared helpers for the GPU parity tests: tolerances and per-sequence oracle results."""
from __future__ import annotations

import numpy as np

import mla_inputs as I
from oracle import mla_oracle as O

F32_TOL = 1e-4   # max |g - o| / max(|o|, RMS(o))
BF16_TOL = 2e-2  # max |g - o| / RMS(o)


def bf16_half_ulp(ref) -> np.ndarray:
    """Half the spacing of bf16 numbers at |ref| (the rounding error of storing ref in bf16)."""
    a = np.abs(np.asarray(ref, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 8), 0.0)


def rel_err(got, ref, dtype: str) -> float:
    """fp32: max |g - o| / max(|o|, RMS(o)).
    bf16: max (|g - o| - half an ulp of o in bf16) / RMS(o): the result is stored in bf16,
    so its own final rounding is not counted against the 2e-2 budget."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    rms = float(np.sqrt(np.mean(ref * ref)))
    if dtype == "f32":
        denom = np.maximum(np.abs(ref), rms)
        return float(np.max(np.abs(got - ref) / denom))
    excess = np.maximum(np.abs(got - ref) - bf16_half_ulp(ref), 0.0)
    return float(np.max(excess) / rms)


def assert_close(got, ref, dtype: str, what: str = ""):
    err = rel_err(got, ref, dtype)
    tol = F32_TOL if dtype == "f32" else BF16_TOL
    assert np.all(np.isfinite(np.asarray(got, dtype=np.float64))), f"{what}: non-finite values"
    assert err <= tol, f"{what}: relative error {err:.3e} > {tol:g}"
    return err


def assert_close_rows(got, ref, what: str = "", tol: float = BF16_TOL):
    """The bf16 measure of rel_err applied to each query token on its own (reading c20): the outputs of
    one prompt's queries average 1..L tokens, so their magnitudes differ by up to sqrt(L) and one
    global RMS would hold the long rows to a loose bound and the short rows to a tight one."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    n = ref.shape[0]
    g, r = got.reshape(n, -1), ref.reshape(n, -1)
    rms = np.sqrt(np.mean(r * r, axis=1))
    excess = np.maximum(np.abs(g - r) - bf16_half_ulp(r), 0.0)
    err = excess.max(axis=1) / rms
    worst = int(np.argmax(err))
    assert err[worst] <= tol, f"{what}: query row {worst}: relative error {err[worst]:.3e} > {tol:g}"
    return float(err[worst])


def logical_cache(p: I.Problem, b: int):
    """Oracle-side cache rows of sequence b (float64): drawn rows or rows projected from x_ctx,
    then the appended query tokens projected from x_q."""
    d = p.dims
    L = int(p.lens[b])
    fp8 = getattr(p.w, "cache_fp8", False)
    if p.w.fill == "direct" and fp8:
        codes, k, kr = I.draw_fp8_rows(p.w, b, L)
        c, k_r = O.dequantize_latent_fp8(O.e4m3_value(codes), 2.0 ** k, kr)
    elif p.w.fill == "direct":
        rows = I.draw_latent_rows(p.w, b, L).astype(np.float64)
        c, k_r = rows[:, :d.d_c], rows[:, d.d_c:]
    else:
        start = int(p.lens[:b].sum())
        c, k_r = O.compress(p.x_ctx[start:start + L], p.weights["W_DKV"], p.weights["W_KR"], np.arange(L), d.rope_base)
        if fp8:
            c, k_r = O.dequantize_latent_fp8(*O.quantize_latent_fp8(c, k_r))
    if p.w.n_append:
        sl = slice(b * p.w.n_q, (b + 1) * p.w.n_q)
        c2, r2 = O.compress(p.x_q[sl], p.weights["W_DKV"], p.weights["W_KR"], p.q_pos[sl], d.rope_base)
        if fp8:
            c2, r2 = O.dequantize_latent_fp8(*O.quantize_latent_fp8(c2, r2))
        c, k_r = np.concatenate([c, c2]), np.concatenate([k_r, r2])
    return c, k_r


def oracle_sequence(p: I.Problem, b: int, explicit: bool = True) -> dict:
    """Everything the oracle says about sequence b of a workload step.

    o_lat / lse are the attention stage's result on the inputs the bf16 method
    stores (cache rows and absorbed queries rounded to bf16 by the oracle's own
    rounding, reading c9); `out` is the pure float64 chain from x."""
    d, W = p.dims, p.weights
    n_q = p.w.n_q
    sl = slice(b * n_q, (b + 1) * n_q)
    c, k_r = logical_cache(p, b)
    q_nope, q_rope = O.project_query(p.x_q[sl], W["W_Q"], W["W_QR"], p.q_pos[sl], d.n_heads, d.rope_base)
    q_abs = O.absorb_query(q_nope, W["W_UK"])
    scale = O.softmax_scale(d.qk_nope, d.d_rope)
    kv = int(p.kv_len[b])
    st = O.round_bf16 if p.w.dtype == "bf16" else (lambda v: v)
    o_lat, lse = O.attend_latent(st(q_abs), st(q_rope), st(c), st(k_r), kv, scale)
    res = dict(c=c, k_r=k_r, q_abs=q_abs, q_rope=q_rope, o_lat=o_lat, lse=lse)
    if explicit:
        o = O.attend_explicit(q_nope, q_rope, c, k_r, W["W_UK"], W["W_UV"], kv, scale)
        res["out"] = O.output_project(o, W["W_O"])
    else:
        o_lat64, _ = O.attend_latent(q_abs, q_rope, c, k_r, kv, scale)
        res["out"] = O.output_project(O.up_project_values(o_lat64, W["W_UV"]), W["W_O"])
    return res


def _bf16_ulp(v):
    v = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(v, 1e-30)))
    return 2.0 ** (e - 7)


def append_c13_masks(x, W_DKV, W_KR, pos, base):
    """Float64 cache rows of x (oracle), the fp32 accumulation bound of each element, and the mask of
    elements whose value lies farther from a bf16 rounding midpoint than that bound (reading c13).

    The bound is a wide estimate of fp32 accumulation error: 16 * 2u * sqrt(K) * ||w * x||_2 with
    u = 2^-24; a rotated RoPE pair mixes both unrotated values and adds the fp32 table and product
    roundings (2^-20 relative).  The mask depends on the inputs and the oracle only, never on the GPU."""
    xs = np.asarray(x, dtype=np.float64)
    c, k_r = O.compress(xs, W_DKV, W_KR, pos, base)
    ref = np.concatenate([c, k_r], axis=1)
    K = xs.shape[1]
    u = 2.0 ** -23 * np.sqrt(K) * 16
    acc_c = u * np.sqrt((xs * xs) @ (np.asarray(W_DKV, dtype=np.float64) ** 2).T)
    y = xs @ np.asarray(W_KR, dtype=np.float64).T
    acc_y = u * np.sqrt((xs * xs) @ (np.asarray(W_KR, dtype=np.float64) ** 2).T)
    pair = acc_y[:, 0::2] + acc_y[:, 1::2] + 2.0 ** -20 * (np.abs(y[:, 0::2]) + np.abs(y[:, 1::2]))
    bound = np.concatenate([acc_c, np.repeat(pair, 2, axis=1)], axis=1)
    ulp = _bf16_ulp(ref)
    lo = np.floor(ref / ulp) * ulp
    safe = np.abs(ref - (lo + ulp / 2)) > bound
    return ref, bound, safe


# Fraction of elements the exactness part of the c13 check covers, measured with append_c13_masks on
# the DeepSeek-V2-shaped layer (Gaussian x, N(0, 1/d_model) weights): 0.822 (64 rows appended at
# position 8191), 0.826 (256 rows at positions up to 32,768), 0.825 (2048 sampled rows of the
# 65,536-token cache build); by part, latent 0.83-0.84 and RoPE key 0.73-0.74 (the rotation adds the
# table and product roundings to the bound).  The check asserts the measured coverage, rounded down,
# so that a change of inputs or bound that quietly empties the exact subset fails instead of passing
# vacuously.
C13_MIN_SAFE_FRACTION = 0.8


def assert_append_c13(got, x, W_DKV, W_KR, pos, base, what=""):
    """Reading c13 on bf16 cache rows `got` [T, d_c + d_rope] appended from x [T, d_model] at `pos`:
    every element within one bf16 ulp plus the accumulation bound of the float64 value, and equal to
    its round-to-nearest-even wherever the float64 value is farther from a midpoint than the bound."""
    ref, bound, safe = append_c13_masks(x, W_DKV, W_KR, pos, base)
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.abs(got - ref) <= _bf16_ulp(ref) + bound), f"{what}: beyond one ulp + accumulation bound"
    frac = float(np.mean(safe))
    assert frac >= C13_MIN_SAFE_FRACTION, f"{what}: exactness check covers only {frac:.3f} of the elements"
    rne = I.round_to_bf16(ref.astype(np.float32)).astype(np.float64)
    bad = np.flatnonzero(got[safe] != rne[safe])
    assert bad.size == 0, f"{what}: {bad.size} elements differ from RNE(oracle) where the rounding is decided"
    return frac
