"""Checks that pin the float64 oracle to things other than itself.

Each ``check_*`` function raises AssertionError when the oracle disagrees
with a brute-force scalar computation, a library routine, an algebraic
invariant, a special case or a closed form the pages print.  The checks are
called by test_oracle.py and, with deliberate mistakes planted in the
oracle, by test_oracle_mutations.py (which expects them to fail).
"""
from __future__ import annotations

import cmath
import json
import math
import os

import numpy as np

from oracle import mla_oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ small random problems
def small_problem(seed, d_model, H, qk_nope, d_rope, v_head, d_c, L, n_q, sharp=1.0):
    rng = np.random.default_rng(seed)
    W = {
        "W_DKV": rng.standard_normal((d_c, d_model)) / math.sqrt(d_model),
        "W_KR": rng.standard_normal((d_rope, d_model)) / math.sqrt(d_model),
        "W_Q": sharp * rng.standard_normal((H * qk_nope, d_model)) / math.sqrt(d_model),
        "W_QR": sharp * rng.standard_normal((H * d_rope, d_model)) / math.sqrt(d_model),
        "W_UK": rng.standard_normal((H, qk_nope, d_c)) / math.sqrt(d_c),
        "W_UV": rng.standard_normal((H, v_head, d_c)) / math.sqrt(d_c),
        "W_O": rng.standard_normal((d_model, H * v_head)) / math.sqrt(H * v_head),
    }
    x_ctx = rng.standard_normal((L, d_model))
    x_q = rng.standard_normal((n_q, d_model))
    return W, x_ctx, x_q


# ------------------------------------------------------------------ brute force (pure Python scalars)
def bf_rotate(vec, pos, base):
    """Rotate pairs (v[2i], v[2i+1]) as the complex number v[2i] + i v[2i+1] times e^{i pos theta_i}."""
    d = len(vec)
    out = [0.0] * d
    for i in range(d // 2):
        theta = base ** (-(2.0 * i) / d)
        z = complex(vec[2 * i], vec[2 * i + 1]) * cmath.exp(1j * pos * theta)
        out[2 * i], out[2 * i + 1] = z.real, z.imag
    return out


def bf_matvec(W, x):
    """y[r] = sum_k W[r][k] x[k] with explicit loops."""
    rows, cols = len(W), len(x)
    return [sum(W[r][k] * x[k] for k in range(cols)) for r in range(rows)]


def bf_decode_layer(W, x_ctx, x_q, H, qk_nope, d_rope, v_head, d_c, kv_len, n_q, base=10000.0):
    """The explicit MLA decode layer, scalar by scalar, written straight from the definitions:
    cache c_t = W_DKV x_t and k_R,t = RoPE(W_KR x_t, t); per head keys
    [W_UK^h c_t || k_R,t] and values W_UV^h c_t; queries [W_Q^h x || RoPE(W_QR^h x, p)];
    softmax over the first vis_j tokens scaled by 1/sqrt(qk_nope + d_rope);
    output W_O times the concatenated head outputs."""
    Wd = W["W_DKV"].tolist(); Wr = W["W_KR"].tolist()
    Wq = W["W_Q"].tolist(); Wqr = W["W_QR"].tolist()
    Wuk = W["W_UK"].tolist(); Wuv = W["W_UV"].tolist(); Wo = W["W_O"].tolist()
    L = len(x_ctx)
    cache_c, cache_r = [], []
    for t in range(L):
        xt = list(map(float, x_ctx[t]))
        cache_c.append(bf_matvec(Wd, xt))
        cache_r.append(bf_rotate(bf_matvec(Wr, xt), t, base))
    scale = 1.0 / math.sqrt(qk_nope + d_rope)
    outs = []
    for j in range(n_q):
        xq = list(map(float, x_q[j]))
        qpos = kv_len - n_q + j          # the query tokens are the last n_q cached positions
        vis = kv_len - (n_q - 1 - j)
        qn_all = bf_matvec(Wq, xq)
        qr_all = bf_matvec(Wqr, xq)
        concat = []
        for h in range(H):
            qn = qn_all[h * qk_nope:(h + 1) * qk_nope]
            qr = bf_rotate(qr_all[h * d_rope:(h + 1) * d_rope], qpos, base)
            scores, values = [], []
            for t in range(vis):
                k_content = [sum(Wuk[h][i][cc] * cache_c[t][cc] for cc in range(d_c)) for i in range(qk_nope)]
                v = [sum(Wuv[h][i][cc] * cache_c[t][cc] for cc in range(d_c)) for i in range(v_head)]
                dot = sum(qn[i] * k_content[i] for i in range(qk_nope)) + sum(qr[i] * cache_r[t][i] for i in range(d_rope))
                scores.append(scale * dot)
                values.append(v)
            if vis == 0:
                concat.extend([0.0] * v_head)
                continue
            mx = max(scores)
            ex = [math.exp(s - mx) for s in scores]
            z = sum(ex)
            concat.extend(sum(ex[t] / z * values[t][i] for t in range(vis)) for i in range(v_head))
        outs.append(bf_matvec(Wo, concat))
    return np.array(outs), np.array(cache_c), np.array(cache_r)


def _oracle_layer(W, x_ctx, x_q, H, qk_nope, d_rope, v_head, d_c, kv_len, n_q, base=10000.0):
    from mla_inputs import Dims
    dims = Dims(d_model=x_ctx.shape[1], n_heads=H, qk_nope=qk_nope, d_rope=d_rope,
                v_head=v_head, d_c=d_c, rope_base=base)
    L = x_ctx.shape[0]
    c, k_r = O.compress(x_ctx, W["W_DKV"], W["W_KR"], np.arange(L), base)
    q_pos = np.array([kv_len - n_q + j for j in range(n_q)])
    out = O.decode_layer_explicit(x_q, q_pos, [(c, k_r)], W, dims, n_q, [kv_len])
    return out, c, k_r, dims, q_pos


# ------------------------------------------------------------------ checks
def check_page1_shapes():
    g = _golden("page1_shapes.json")
    rng = np.random.default_rng(0)
    x = rng.standard_normal((g["seq"], g["d_model"]))
    W_DKV = rng.standard_normal((g["d_latent"], g["d_model"]))
    W_KR = rng.standard_normal((16, g["d_model"]))
    W_UK = rng.standard_normal((g["n_heads"], g["d_head"], g["d_latent"]))
    W_UV = rng.standard_normal((g["n_heads"], g["d_head"], g["d_latent"]))
    c, _ = O.compress(x, W_DKV, W_KR, np.arange(g["seq"]))
    assert list(c.shape) == g["latent_shape"]
    keys = np.stack([O.reconstruct_kv(c, W_UK, W_UV, h)[0] for h in range(g["n_heads"])], axis=1)
    assert list(keys.shape) == g["keys_shape"]


def check_bruteforce(seed, d_model, H, qk_nope, d_rope, v_head, d_c, L, n_q, tol=1e-12):
    W, x_ctx, x_q = small_problem(seed, d_model, H, qk_nope, d_rope, v_head, d_c, L, n_q)
    kv_len = L
    bf_out, bf_c, bf_r = bf_decode_layer(W, x_ctx, x_q, H, qk_nope, d_rope, v_head, d_c, kv_len, n_q)
    out, c, k_r, _, _ = _oracle_layer(W, x_ctx, x_q, H, qk_nope, d_rope, v_head, d_c, kv_len, n_q)
    for got, ref in ((c, bf_c), (k_r, bf_r), (out, bf_out)):
        err = np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-300)
        assert err <= tol, err


def check_absorbed_equals_explicit(seed, d_model, H, qk_nope, d_rope, v_head, d_c, L, n_q, tol=1e-10):
    W, x_ctx, x_q = small_problem(seed, d_model, H, qk_nope, d_rope, v_head, d_c, L, n_q, sharp=3.0)
    out, c, k_r, dims, q_pos = _oracle_layer(W, x_ctx, x_q, H, qk_nope, d_rope, v_head, d_c, L, n_q)
    out_abs = O.decode_layer_absorbed(x_q, q_pos, [(c, k_r)], W, dims, n_q, [L])
    err = np.max(np.abs(out - out_abs)) / np.max(np.abs(out))
    assert err <= tol, err


def check_sdpa(seed, d_model, H, qk_nope, d_rope, v_head, d_c, L, n_q, tol=1e-12):
    """torch's scaled_dot_product_attention (CPU, float64) over the oracle's rebuilt K and V."""
    import torch
    W, x_ctx, x_q = small_problem(seed, d_model, H, qk_nope, d_rope, v_head, d_c, L, n_q, sharp=2.0)
    c, k_r = O.compress(x_ctx, W["W_DKV"], W["W_KR"], np.arange(L))
    q_pos = np.array([L - n_q + j for j in range(n_q)])
    q_nope, q_rope = O.project_query(x_q, W["W_Q"], W["W_QR"], q_pos, H)
    scale = O.softmax_scale(qk_nope, d_rope)
    got = O.attend_explicit(q_nope, q_rope, c, k_r, W["W_UK"], W["W_UV"], L, scale)
    K = np.stack([np.concatenate([O.reconstruct_kv(c, W["W_UK"], W["W_UV"], h)[0], k_r], axis=1) for h in range(H)])
    V = np.stack([O.reconstruct_kv(c, W["W_UK"], W["W_UV"], h)[1] for h in range(H)])
    Q = np.concatenate([q_nope, q_rope], axis=2).transpose(1, 0, 2)          # [H, n_q, 192]
    mask = np.zeros((n_q, L), dtype=bool)
    for j in range(n_q):
        mask[j, :O.visible(L, n_q, j)] = True
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Q)[None], torch.from_numpy(K)[None], torch.from_numpy(V)[None],
        attn_mask=torch.from_numpy(mask), scale=scale)[0].numpy().transpose(1, 0, 2)
    err = np.max(np.abs(got - ref)) / np.max(np.abs(ref))
    assert err <= tol, err


def check_per_head_rope(seed=13, d_model=48, H=3, qk_nope=5, d_rope=4, v_head=6, d_c=7, L=11):
    """The per-head positional keys: with every head's W_KR^h equal to one W_KR the keys and the result
    equal the shared-key ones; with different heads, torch's scaled_dot_product_attention (float64) over
    K^h = [W_UK^h c || k_R^h] agrees with attend_explicit_at; the rotation restarts per head (head h's
    key equals the shared rotation of its own rows)."""
    import torch
    pos = np.arange(L - 4, L)
    W, x_ctx, x_q = small_problem(seed, d_model, H, qk_nope, d_rope, v_head, d_c, L, len(pos), sharp=2.0)
    W_KR_h = np.random.default_rng(seed + 1).standard_normal((H * d_rope, d_model)) / math.sqrt(d_model)
    c1, k1 = O.compress(x_ctx, W["W_DKV"], W["W_KR"], np.arange(L))
    c2, k2 = O.compress_per_head_rope(x_ctx, W["W_DKV"], np.tile(W["W_KR"], (H, 1)), np.arange(L), H)
    assert np.allclose(c1, c2) and all(np.allclose(k2[:, h], k1, atol=1e-13) for h in range(H))
    for h in range(H):
        _, kh = O.compress(x_ctx, W["W_DKV"], W_KR_h[h * d_rope:(h + 1) * d_rope], np.arange(L))
        _, kall = O.compress_per_head_rope(x_ctx, W["W_DKV"], W_KR_h, np.arange(L), H)
        assert np.allclose(kall[:, h], kh, atol=1e-13)
    q_nope, q_rope = O.project_query(x_q, W["W_Q"], W["W_QR"], pos, H)
    scale = O.softmax_scale(qk_nope, d_rope)
    s1, _ = O.attend_explicit_at(q_nope, q_rope, pos, c1, k1, W["W_UK"], W["W_UV"], scale)
    s2, _ = O.attend_explicit_at(q_nope, q_rope, pos, c2, k2, W["W_UK"], W["W_UV"], scale)
    assert np.max(np.abs(s1 - s2)) <= 1e-12
    _, kall = O.compress_per_head_rope(x_ctx, W["W_DKV"], W_KR_h, np.arange(L), H)
    got, _ = O.attend_explicit_at(q_nope, q_rope, pos, c1, kall, W["W_UK"], W["W_UV"], scale)
    K = np.stack([np.concatenate([O.reconstruct_kv(c1, W["W_UK"], W["W_UV"], h)[0], kall[:, h]], axis=1) for h in range(H)])
    V = np.stack([O.reconstruct_kv(c1, W["W_UK"], W["W_UV"], h)[1] for h in range(H)])
    Q = np.concatenate([q_nope, q_rope], axis=2).transpose(1, 0, 2)
    mask = np.arange(L)[None, :] <= pos[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Q)[None], torch.from_numpy(K)[None], torch.from_numpy(V)[None],
        attn_mask=torch.from_numpy(mask), scale=scale)[0].numpy().transpose(1, 0, 2)
    assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) <= 1e-12
    out_e = O.attend_explicit(q_nope, q_rope, c1, kall, W["W_UK"], W["W_UV"], L, scale)
    assert np.max(np.abs(out_e - got)) <= 1e-12


def check_prefill_rows(seed, d_model, H, qk_nope, d_rope, v_head, d_c, L, pos, tol=1e-12):
    """attend_explicit_at against torch's scaled_dot_product_attention (CPU, float64) with the
    prompt's causal mask over the rebuilt K and V; its lse against the absorbed form's (the pages'
    invariant: scores are the same either way)."""
    import torch
    pos = np.asarray(pos)
    n = len(pos)
    W, x_ctx, x_q = small_problem(seed, d_model, H, qk_nope, d_rope, v_head, d_c, L, n, sharp=2.0)
    c, k_r = O.compress(x_ctx, W["W_DKV"], W["W_KR"], np.arange(L))
    q_nope, q_rope = O.project_query(x_q, W["W_Q"], W["W_QR"], pos, H)
    scale = O.softmax_scale(qk_nope, d_rope)
    got, lse = O.attend_explicit_at(q_nope, q_rope, pos, c, k_r, W["W_UK"], W["W_UV"], scale)
    K = np.stack([np.concatenate([O.reconstruct_kv(c, W["W_UK"], W["W_UV"], h)[0], k_r], axis=1) for h in range(H)])
    V = np.stack([O.reconstruct_kv(c, W["W_UK"], W["W_UV"], h)[1] for h in range(H)])
    Q = np.concatenate([q_nope, q_rope], axis=2).transpose(1, 0, 2)
    mask = np.arange(L)[None, :] <= pos[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Q)[None], torch.from_numpy(K)[None], torch.from_numpy(V)[None],
        attn_mask=torch.from_numpy(mask), scale=scale)[0].numpy().transpose(1, 0, 2)
    err = np.max(np.abs(got - ref)) / np.max(np.abs(ref))
    assert err <= tol, err
    q_abs = O.absorb_query(q_nope, W["W_UK"])
    for j in range(n):
        _, lse_abs = O.attend_latent(q_abs[j:j + 1], q_rope[j:j + 1], c, k_r, int(pos[j]) + 1, scale)
        assert np.max(np.abs(lse[j] - lse_abs[0])) <= 1e-10


def check_fp8_format(seed=12):
    """The reduced-precision cache format (reading c21) against torch's float8_e4m3fn: rounding of
    50,000 values over the whole range (with exact ties and subnormals), the value of every bit
    pattern, and the scale rule (max |c| / s in (224, 448], s a power of two)."""
    import torch
    rng = np.random.default_rng(seed)
    x = np.concatenate([
        rng.uniform(-448, 448, 20000),
        np.sign(rng.standard_normal(20000)) * 2.0 ** rng.uniform(-12, 8.8, 20000),
        # exact ties: midpoints between neighbouring codes (normal and subnormal)
        (np.arange(1, 64) + 0.5) * 2.0 ** -9, (8 + np.arange(0, 8) + 0.5) * 2.0 ** -3 * 2.0 ** 4,
        [0.0, 448.0, -448.0, 2.0 ** -6, 2.0 ** -9, 1.5 * 2.0 ** -10],
    ])
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    exact32 = x.astype(np.float32).astype(np.float64) == x     # torch converts from float32
    got = O.round_e4m3(x)
    assert np.array_equal(got[exact32], ref[exact32])
    codes = np.arange(256, dtype=np.uint8)
    tv = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ov = O.e4m3_value(codes)
    assert np.array_equal(np.isnan(ov), np.isnan(tv)) and np.array_equal(ov[~np.isnan(ov)], tv[~np.isnan(tv)])
    rows = rng.standard_normal((500, 64)) * 2.0 ** rng.uniform(-30, 30, (500, 1))
    sc = O.fp8_token_scale(rows)
    ratio = np.max(np.abs(rows), axis=1) / sc
    assert np.all(ratio <= 448) and np.all(ratio > 224)
    assert np.all(np.log2(sc) == np.round(np.log2(sc)))
    assert O.fp8_token_scale(np.zeros((1, 8)))[0] == 1.0
    # round trip: every code of the row's range stands for itself; the error is at most half a spacing
    codes_v, s, _ = O.quantize_latent_fp8(rows, rows[:, :4])
    assert np.all(np.abs(codes_v) <= 448)
    err = np.abs(codes_v * s[:, None] - rows)
    assert np.all(err <= 2.0 ** -4 * np.abs(rows) + 2.0 ** -10 * s[:, None])
    # the stored positional key: (k_R / s) rounded to bf16, times s, is k_R within half a bf16 ulp
    keys = rng.standard_normal((500, 16)) * 2.0 ** rng.uniform(-5, 5, (500, 1))
    _, s2, krs = O.quantize_latent_fp8(rows, keys)
    _, k_back = O.dequantize_latent_fp8(np.zeros_like(rows), s2, krs)
    assert np.all(np.abs(k_back - keys) <= 2.0 ** -8 * np.abs(keys))


def check_rope_properties(d_rope=16, base=10000.0):
    rng = np.random.default_rng(7)
    v = rng.standard_normal((5, d_rope))
    # identity at position 0
    assert np.array_equal(O.apply_rope(v, np.zeros(5), base), v)
    # norm preserved
    for p in (1, 17, 4095, 65535):
        r = O.apply_rope(v, np.full(5, p), base)
        assert np.allclose(np.linalg.norm(r, axis=1), np.linalg.norm(v, axis=1), rtol=1e-13)
    # scores depend only on the position difference
    q, k = rng.standard_normal(d_rope), rng.standard_normal(d_rope)
    for p, t, delta in ((10, 3, 100), (7, 7, 12345), (0, 50, 999)):
        a = O.apply_rope(q, p + delta, base) @ O.apply_rope(k, t + delta, base)
        b = O.apply_rope(q, p, base) @ O.apply_rope(k, t, base)
        assert abs(a - b) <= 1e-9 * (1 + abs(b)), (a, b)
    # d_rope = 2: the textbook 2x2 rotation by pos radians
    for p in (0.0, 1.0, 2.5, 1000.0):
        w = np.array([0.3, -1.7])
        R = np.array([[math.cos(p), -math.sin(p)], [math.sin(p), math.cos(p)]])
        assert np.allclose(O.apply_rope(w, p, base), R @ w, rtol=0, atol=1e-12)
    # agrees with rotation written as complex multiplication, on every pair
    for p in (3, 1234):
        assert np.allclose(O.apply_rope(v[0], p, base), bf_rotate(list(v[0]), p, base), rtol=0, atol=1e-12)


def check_special_cases(seed=11, d_model=64, H=4, qk_nope=16, d_rope=8, v_head=12, d_c=20):
    scale = O.softmax_scale(qk_nope, d_rope)
    W, x_ctx, x_q = small_problem(seed, d_model, H, qk_nope, d_rope, v_head, d_c, 9, 1)
    c, k_r = O.compress(x_ctx, W["W_DKV"], W["W_KR"], np.arange(9))
    q_nope, q_rope = O.project_query(x_q, W["W_Q"], W["W_QR"], [9], H)
    # one visible token: every head returns that token's value
    o1 = O.attend_explicit(q_nope, q_rope, c[:1], k_r[:1], W["W_UK"], W["W_UV"], 1, scale)
    for h in range(H):
        assert np.allclose(o1[0, h], W["W_UV"][h] @ c[0], rtol=1e-13, atol=1e-14)
    # identical cached rows: output does not depend on the query
    cc, rr = np.repeat(c[:1], 9, axis=0), np.repeat(k_r[:1], 9, axis=0)
    oa = O.attend_explicit(q_nope, q_rope, cc, rr, W["W_UK"], W["W_UV"], 9, scale)
    ob = O.attend_explicit(5 * q_nope + 1, -q_rope, cc, rr, W["W_UK"], W["W_UV"], 9, scale)
    assert np.allclose(oa, ob, rtol=1e-12, atol=1e-14)
    # zero query: uniform average of the values
    oz = O.attend_explicit(0 * q_nope, 0 * q_rope, c, k_r, W["W_UK"], W["W_UV"], 9, scale)
    for h in range(H):
        assert np.allclose(oz[0, h], (W["W_UV"][h] @ c.T).mean(axis=1), rtol=1e-12, atol=1e-14)
    # very sharp query: one-hot on the highest-scoring token
    big = 1e3
    os_ = O.attend_explicit(big * q_nope, big * q_rope, c, k_r, W["W_UK"], W["W_UV"], 9, scale)
    for h in range(H):
        s = c @ W["W_UK"][h].T @ q_nope[0, h] + k_r @ q_rope[0, h]
        assert np.allclose(os_[0, h], W["W_UV"][h] @ c[int(np.argmax(s))], rtol=1e-9, atol=1e-12)
    # causal pair: query 0 of two equals a single-token decode over one fewer token
    W2, x_ctx2, x_q2 = small_problem(seed + 1, d_model, H, qk_nope, d_rope, v_head, d_c, 8, 2)
    c2, r2 = O.compress(x_ctx2, W2["W_DKV"], W2["W_KR"], np.arange(8))
    qn2, qr2 = O.project_query(x_q2, W2["W_Q"], W2["W_QR"], [6, 7], H)
    pair = O.attend_explicit(qn2, qr2, c2, r2, W2["W_UK"], W2["W_UV"], 8, scale)
    single0 = O.attend_explicit(qn2[:1], qr2[:1], c2[:7], r2[:7], W2["W_UK"], W2["W_UV"], 7, scale)
    single1 = O.attend_explicit(qn2[1:], qr2[1:], c2, r2, W2["W_UK"], W2["W_UV"], 8, scale)
    assert np.allclose(pair[0], single0[0], rtol=1e-13, atol=1e-15)
    assert np.allclose(pair[1], single1[0], rtol=1e-13, atol=1e-15)
    # empty visible set: zero output and -inf log-sum-exp
    q_abs = O.absorb_query(q_nope, W["W_UK"])
    z, lse = O.attend_latent(q_abs, q_rope, c, k_r, 0, scale)
    assert np.all(z == 0) and np.all(np.isneginf(lse))


def check_merge_partials(seed=5, H=4, d_c=24, d_rope=8, L=37):
    rng = np.random.default_rng(seed)
    q_abs, q_r = rng.standard_normal((1, H, d_c)), rng.standard_normal((1, H, d_rope))
    c, k_r = rng.standard_normal((L, d_c)), rng.standard_normal((L, d_rope))
    scale = 0.3
    whole, lse_w = O.attend_latent(q_abs, q_r, c, k_r, L, scale)
    cuts = [0, 5, 6, 30, L]
    parts, lses = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        o, l = O.attend_latent(q_abs, q_r, c[a:b], k_r[a:b], b - a, scale)
        parts.append(o); lses.append(l)
    # an empty part contributes nothing
    o_e, l_e = O.attend_latent(q_abs, q_r, c[:0], k_r[:0], 0, scale)
    parts.append(o_e); lses.append(l_e)
    m, lse_m = O.merge_partials(np.stack(parts), np.stack(lses))
    assert np.allclose(m, whole, rtol=1e-13, atol=1e-14)
    assert np.allclose(lse_m, lse_w, rtol=1e-13)
    # lse is the log of the softmax normaliser: check against a direct sum for one head
    s = scale * (c @ q_abs[0, 0] + k_r @ q_r[0, 0])
    assert abs(lse_w[0, 0] - math.log(sum(math.exp(v) for v in s))) < 1e-12


def check_cache_closed_forms():
    g = _golden("cache_sizes.json")
    ex = g["gqa_worked_example"]
    per_tok = O.cache_bytes(1, O.kv_cache_elems_per_token(ex["n_kv_heads"], ex["d_head"], ex["n_layers"]),
                            ex["bytes_per_value"])
    assert per_tok == ex["bytes_per_token"]
    gib = O.cache_bytes(ex["n_tokens"], per_tok // ex["bytes_per_value"], ex["bytes_per_value"]) / 2**30
    assert round(gib, 2) == ex["gib_at_n_tokens"]
    mha = g["mha_128x128"]
    n = O.kv_cache_elems_per_token(mha["n_heads"], mha["d_head"])
    assert n > mha["more_than"] and n == 32768
    d_c = g["mla_latent_width"]["d_c"]
    assert d_c < O.kv_cache_elems_per_token(mha["n_heads"], mha["d_head"])
    mla = O.mla_cache_elems_per_token(d_c, 64)
    assert mla == 576 and abs(n / mla - 56.888) < 1e-3
    assert O.mla_cache_elems_per_token(64, 16) == 80 and O.kv_cache_elems_per_token(8, 64) == 1024


def check_round_bf16():
    """The oracle's bf16 rounding against torch's float -> bfloat16 conversion and hand-made ties."""
    import torch
    rng = np.random.default_rng(9)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 6, 20000), [0.0, -0.0, 1.0, -3.0]])
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    # torch rounds the float32 value; compare on inputs that are exact in float32
    x32 = x.astype(np.float32).astype(np.float64)
    assert np.array_equal(O.round_bf16(x32), ref)
    # ties: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 -> even (1); 1 + 3*2^-8 -> 1 + 2^-6
    assert O.round_bf16(np.array([1 + 2.0 ** -8]))[0] == 1.0
    assert O.round_bf16(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6
    assert O.round_bf16(np.array([-(1 + 2.0 ** -8 + 2.0 ** -20)]))[0] == -(1 + 2.0 ** -7)
