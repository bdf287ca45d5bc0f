"""Shared helpers for the GPU parity tests: tolerances and per-sequence oracle results."""
from __future__ import annotations

import numpy as np

import mla_inputs as I
from oracle import mla_oracle as O

F32_TOL = 1e-4   # max |g - o| / max(|o|, RMS(o))
BF16_TOL = 2e-2  # max |g - o| / RMS(o)


def rel_err(got, ref, dtype: str) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    rms = float(np.sqrt(np.mean(ref * ref)))
    if dtype == "f32":
        denom = np.maximum(np.abs(ref), rms)
        return float(np.max(np.abs(got - ref) / denom))
    return float(np.max(np.abs(got - ref)) / rms)


def assert_close(got, ref, dtype: str, what: str = ""):
    err = rel_err(got, ref, dtype)
    tol = F32_TOL if dtype == "f32" else BF16_TOL
    assert np.all(np.isfinite(np.asarray(got, dtype=np.float64))), f"{what}: non-finite values"
    assert err <= tol, f"{what}: relative error {err:.3e} > {tol:g}"
    return err


def logical_cache(p: I.Problem, b: int):
    """Oracle-side cache rows of sequence b (float64): drawn rows or rows projected from x_ctx,
    then the appended query tokens projected from x_q."""
    d = p.dims
    L = int(p.lens[b])
    if p.w.fill == "direct":
        rows = I.draw_latent_rows(p.w, b, L).astype(np.float64)
        c, k_r = rows[:, :d.d_c], rows[:, d.d_c:]
    else:
        start = int(p.lens[:b].sum())
        c, k_r = O.compress(p.x_ctx[start:start + L], p.weights["W_DKV"], p.weights["W_KR"], np.arange(L), d.rope_base)
    if p.w.n_append:
        sl = slice(b * p.w.n_q, (b + 1) * p.w.n_q)
        c2, r2 = O.compress(p.x_q[sl], p.weights["W_DKV"], p.weights["W_KR"], p.q_pos[sl], d.rope_base)
        c, k_r = np.concatenate([c, c2]), np.concatenate([k_r, r2])
    return c, k_r


def oracle_sequence(p: I.Problem, b: int, explicit: bool = True) -> dict:
    """Everything the oracle says about sequence b of a workload step."""
    d, W = p.dims, p.weights
    n_q = p.w.n_q
    sl = slice(b * n_q, (b + 1) * n_q)
    c, k_r = logical_cache(p, b)
    q_nope, q_rope = O.project_query(p.x_q[sl], W["W_Q"], W["W_QR"], p.q_pos[sl], d.n_heads, d.rope_base)
    q_abs = O.absorb_query(q_nope, W["W_UK"])
    scale = O.softmax_scale(d.qk_nope, d.d_rope)
    kv = int(p.kv_len[b])
    o_lat, lse = O.attend_latent(q_abs, q_rope, c, k_r, kv, scale)
    res = dict(c=c, k_r=k_r, q_abs=q_abs, q_rope=q_rope, o_lat=o_lat, lse=lse)
    if explicit:
        o = O.attend_explicit(q_nope, q_rope, c, k_r, W["W_UK"], W["W_UV"], kv, scale)
        res["out"] = O.output_project(o, W["W_O"])
    else:
        res["out"] = O.output_project(O.up_project_values(o_lat, W["W_UV"]), W["W_O"])
    return res
