"""The reduced-precision latent cache (reading c21: FP8 E4M3 latent codes with one power-of-two scale
per token, the positional key stored in bf16 divided by that scale) against the float64 oracle:

  * the append: scales, codes and stored keys of 197 appended tokens against the oracle's quantiser of
    its own float64 rows; placement exact (every other byte keeps its 0xFF sentinel);
  * the decode step over drawn and over appended reduced-precision caches, o_lat / lse against the
    absorbed oracle on the dequantised rows (the values the method stores, reading c15) and the layer
    output against the explicit float64 chain;
  * prefill over a reduced-precision cache, from hidden states.

Where floating point decides an integer (a code, a scale exponent), the two sides may disagree only
when the float64 value lies within the fp32 accumulation bound of the decision boundary (the bound of
reading c13); there the GPU's code is within one code spacing.  Over a cache the GPU quantised, the
attention check allows for those codes (reading c21): the oracle marks every code within the bound of
a midpoint, recomputes its attention with that code switched to the other neighbour, and the sum of
these effects is added to the tolerance of each output element; everything else is compared as usual."""
import numpy as np
import pytest
import torch

import mla_harness as Hn
import mla_inputs as I
import mla_latent_kv_81_b300 as M
from gpu_helpers import append_c13_masks, assert_close, assert_close_rows, oracle_sequence
from oracle import mla_oracle as O

pytestmark = pytest.mark.gpu


def _status_clean(L):
    code, flags = L.status()
    assert code == 0, (M.mla_status_string(code), flags)


def test_fp8_append_scales_codes_keys_and_placement():
    w = I.Workload("fp8_append", I.DSV2, "bf16", 2, 130, 130, 1, 0, 71, "append", cache_fp8=True)
    p = I.make_problem(w)
    L = Hn.DeviceLayer(p)
    T = 197
    rng = np.random.default_rng(5)
    x = I.draw_hidden(rng, T, I.DSV2.d_model, "bf16")
    seq = np.concatenate([np.zeros(130, np.int32), np.ones(T - 130, np.int32)])
    pos = np.concatenate([np.arange(130), rng.permutation(130)[:T - 130]]).astype(np.int32)
    ws = M.workspace(M.mla_compress_workspace_bytes(L.cfg, T), "cuda")
    M.mla_compress_append(L.cfg, Hn.to_dev(x, "bf16"), L.W["W_DKV"], L.W["W_KR"], torch.from_numpy(seq).cuda(),
                          torch.from_numpy(pos).cuda(), L.rope, L.cache, ws=ws)
    torch.cuda.synchronize()
    code, flags = M.mla_get_device_status(ws)
    assert code == 0, flags
    W = p.weights
    ref, bound, safe_bf16 = append_c13_masks(x, W["W_DKV"], W["W_KR"], pos, I.DSV2.rope_base)
    d_c = I.DSV2.d_c
    c, kr = ref[:, :d_c], ref[:, d_c:]
    codes, kr_s, s = L.cache_rows_at(seq, pos)
    # scales: equal unless the row maximum sits within its accumulation bound of a boundary 448 * 2^k
    s_ref = O.fp8_token_scale(c)
    m = np.abs(c).max(axis=1)
    mb = bound[np.arange(T), np.abs(c).argmax(axis=1)]
    near = (np.abs(m - 448 * s_ref) <= mb) | (np.abs(m - 224 * s_ref) <= mb)
    assert np.all((s == s_ref) | near), np.flatnonzero((s != s_ref) & ~near)[:5]
    same = s == s_ref
    # codes of rows with equal scales: the oracle's rounding wherever c / s lies farther from an E4M3
    # midpoint than the accumulation bound; within one code spacing everywhere
    v = c / s_ref[:, None]
    a = np.abs(v)
    qs = 2.0 ** (np.maximum(np.floor(np.log2(np.where(a > 0, a, 1.0))), -6.0) - 3.0)
    dist = np.abs(a - (np.floor(a / qs) + 0.5) * qs)
    safe = dist > bound[:, :d_c] / s_ref[:, None]
    got = O.e4m3_value(codes)
    want = O.round_e4m3(v)
    sel = safe & same[:, None]
    assert np.array_equal(got[sel], want[sel])
    assert np.all(np.abs(got - want)[same] <= qs[same])
    assert sel.mean() > 0.9 * same.mean()
    # the positional key: (k_R / s) * s is the bf16 rounding of k_R (reading c13 on the key columns)
    kr_g = kr_s * s[:, None]
    ref_k = O.round_bf16(kr)
    sk = safe_bf16[:, d_c:] & same[:, None]
    assert np.array_equal(kr_g[sk], ref_k[sk])
    assert np.all(np.abs(kr_g - ref_k) <= 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref_k), 1e-30))) - 7) + 1e-30)
    # placement: exactly the written slots changed
    codes_v, kr_v, sc_v = L.fp8_parts()
    written = np.zeros((p.num_blocks, I.DSV2.block_size), bool)
    written[p.block_table[seq, pos // 64], pos % 64] = True
    cv = codes_v.cpu().numpy()
    assert np.all(cv.transpose(0, 2, 1)[~written] == 255)
    assert np.all(np.isnan(sc_v.cpu().numpy()[~written]))
    assert not np.any(np.isnan(sc_v.cpu().numpy()[written]))


def ambiguous_code_effects(p: I.Problem, b: int, ref: dict):
    """Elementwise sum, over the codes of sequence b the oracle finds within the fp32 accumulation bound
    of an E4M3 midpoint, of |change of the oracle's o_lat| when that code takes the other neighbour."""
    d, W = p.dims, p.weights
    n = int(p.kv_len[b])
    start, Lb = int(p.lens[:b].sum()), int(p.lens[b])
    x = np.concatenate([p.x_ctx[start:start + Lb], p.x_q[b * p.w.n_q:(b + 1) * p.w.n_q]])
    rows, bound, _ = append_c13_masks(x, W["W_DKV"], W["W_KR"], np.arange(n), d.rope_base)
    c, k_r = rows[:, :d.d_c], rows[:, d.d_c:]
    codes, s, krs = O.quantize_latent_fp8(c, k_r)
    v = c / s[:, None]
    a = np.abs(v)
    qs = 2.0 ** (np.maximum(np.floor(np.log2(np.where(a > 0, a, 1.0))), -6.0) - 3.0)
    mid = (np.floor(a / qs) + 0.5) * qs
    amb = np.argwhere(np.abs(a - mid) <= bound[:, :d.d_c] / s[:, None])
    cq, kq = O.dequantize_latent_fp8(codes, s, krs)
    allow = np.zeros_like(ref["o_lat"])
    scale = O.softmax_scale(d.qk_nope, d.d_rope)
    qa, qr = O.round_bf16(ref["q_abs"]), O.round_bf16(ref["q_rope"])
    for t, e in amb:
        other = np.sign(v[t, e]) * (2 * mid[t, e] - np.abs(codes[t, e]))   # the other neighbour of the midpoint
        c2 = cq.copy()
        c2[t, e] = other * s[t]
        o2, _ = O.attend_latent(qa, qr, c2, kq, n, scale)
        allow += np.abs(o2 - ref["o_lat"])
    return allow, len(amb)


@pytest.mark.parametrize("fill", ["direct", "append"])
def test_fp8_decode_step_matches_the_oracle(fill):
    w = I.Workload(f"fp8_step_{fill}", I.DSV2, "bf16", 3, 100, 700, 1, 1, 72 if fill == "direct" else 73, fill,
                   cache_fp8=True)
    p = I.make_problem(w)
    L = Hn.DeviceLayer(p)
    L.fill()
    L.step()
    torch.cuda.synchronize()
    _status_clean(L)
    o_lat, lse, out = L.o_lat.float().cpu().numpy(), L.lse.cpu().numpy(), L.out.float().cpu().numpy()
    for b in range(w.batch):
        ref = oracle_sequence(p, b, explicit=True)
        if fill == "append":
            allow, n_amb = ambiguous_code_effects(p, b, ref)
            rms = np.sqrt(np.mean(ref["o_lat"] ** 2))
            from gpu_helpers import bf16_half_ulp
            excess = np.maximum(np.abs(o_lat[b:b + 1] - ref["o_lat"]) - bf16_half_ulp(ref["o_lat"]) - allow, 0.0)
            assert excess.max() / rms <= 2e-2, f"o_lat b={b}: {excess.max() / rms:.3e} with {n_amb} ambiguous codes"
        else:
            assert_close(o_lat[b:b + 1], ref["o_lat"], "bf16", f"{fill} o_lat b={b}")
            assert_close(out[b:b + 1], ref["out"], "bf16", f"{fill} out b={b}")
        assert np.max(np.abs(lse[b:b + 1] - ref["lse"])) <= 1e-2


def test_fp8_prefill_from_hidden_states():
    c = I.PREFILL_CASES["prefill_dsv2_L333_T200_x_fp8"]
    p = I.make_prefill(c)
    d, W = p.dims, p.weights
    L = Hn.PrefillLayer(p)
    L.fill()
    L.run()
    torch.cuda.synchronize()
    code, flags = L.status()
    assert code == 0, flags
    cc, k_r = O.compress(p.x, W["W_DKV"], W["W_KR"], np.arange(c.prompt), d.rope_base)
    cq, kq = O.dequantize_latent_fp8(*O.quantize_latent_fp8(cc, k_r))
    xq = p.x[c.prompt - c.queries:]
    ref = O.decode_layer_explicit(xq, p.q_pos, [(cq, kq)], W, d, c.queries, [c.prompt])
    assert_close_rows(L.out.float().cpu().numpy(), ref, "fp8 prefill out")
