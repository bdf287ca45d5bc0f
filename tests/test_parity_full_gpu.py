"""Full-size workloads (the DeepSeek-V2-shaped layer at its benchmark sizes) run through the same
decode step the benchmark times, then checked against the float64 oracle:

  * o_lat and lse of every query of every sequence, against the absorbed form (identical to the
    explicit form in float64, pinned by the invariant test), on the stored bf16 inputs (reading c15);
  * the layer output of three sequences (shortest, longest, one drawn at random) against the pure
    float64 explicit chain from x (K and V rebuilt per head);
  * every appended cache row with reading c13 (exact where the rounding is decided, within one ulp plus
    the accumulation bound elsewhere), and for the cache built by appending 65,536 tokens a seeded
    sample of 2048 of its rows."""
import numpy as np
import pytest
import torch

import mla_harness as Hn
import mla_inputs as I
import mla_latent_kv_81_b300 as M
from gpu_helpers import assert_append_c13, assert_close, logical_cache, oracle_sequence
from oracle import mla_oracle as O

pytestmark = pytest.mark.gpu

FULL = ["dsv2_b16_ctx4096", "dsv2_b64_ctx1k_8k", "dsv2_b64_ctx8192", "dsv2_b4_ctx65536",
        "dsv2_b128_ctx4k_32k_nq2", "dsv2_b64_ctx8192_fp8"]


def assert_fp8_rows_close(got, x, W_DKV, W_KR, pos, base, what):
    """Reduced-precision rows read back (codes, k_R / s, s) against the oracle's quantiser of its own
    float64 rows: the dequantised latent within one code spacing times the scale (a code or scale may
    differ from the oracle's where the float64 value lies within fp32 rounding of a decision
    boundary; test_fp8_gpu checks the exact cases), the positional key within one bf16 ulp."""
    codes, kr_s, s = got
    c, k_r = O.compress(np.asarray(x, dtype=np.float64), W_DKV, W_KR, pos, base)
    cq, kq = O.dequantize_latent_fp8(*O.quantize_latent_fp8(c, k_r))
    cg = O.e4m3_value(codes) * s[:, None]
    assert np.all(np.isfinite(cg)), what
    smax = np.maximum(s, O.fp8_token_scale(c))[:, None]
    spacing = 2.0 ** (np.maximum(np.floor(np.log2(np.maximum(np.abs(cq) / smax, 1e-30))), -6.0) - 3.0) * smax
    assert np.all(np.abs(cg - cq) <= spacing + 1e-30), what
    kg = kr_s * s[:, None]
    assert np.all(np.abs(kg - kq) <= 2.0 ** (np.floor(np.log2(np.maximum(np.abs(kq), 1e-30))) - 7) + 1e-30), what


def samples(p: I.Problem):
    lens = p.kv_len
    picks = [int(np.argmin(lens)), int(np.argmax(lens)), int(np.random.default_rng(p.w.seed).integers(p.w.batch))]
    return sorted(set(picks))


@pytest.mark.parametrize("name", FULL)
def test_full_size_step(name):
    p = I.make_problem(I.WORKLOADS[name])
    d, W = p.dims, p.weights
    L = Hn.DeviceLayer(p)
    L.fill()
    L.step()
    torch.cuda.synchronize()
    code, flags = L.status()
    assert code == 0, (M.mla_status_string(code), flags)
    out = L.out.float().cpu().numpy()
    o_lat = L.o_lat.float().cpu().numpy()
    lse = L.lse.cpu().numpy()
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(o_lat)) and np.all(np.isfinite(lse))
    n_q, H = p.w.n_q, d.n_heads

    # attention stage, every sequence: the oracle's queries for the whole batch at once
    q_nope, q_rope = O.project_query(p.x_q, W["W_Q"], W["W_QR"], p.q_pos, H, d.rope_base)
    q_abs = O.absorb_query(q_nope, W["W_UK"])
    qa, qr = O.round_bf16(q_abs), O.round_bf16(q_rope)
    scale = O.softmax_scale(d.qk_nope, d.d_rope)
    for b in range(p.w.batch):
        c, k_r = logical_cache(p, b)
        # the rows the method stores: projected rows rounded to bf16 (drawn rows already are bf16)
        k0 = 0 if p.w.fill == "append" else int(p.lens[b])
        c[k0:], k_r[k0:] = O.round_bf16(c[k0:]), O.round_bf16(k_r[k0:])
        sl = slice(b * n_q, (b + 1) * n_q)
        ref_o, ref_lse = O.attend_latent(qa[sl], qr[sl], c, k_r, int(p.kv_len[b]), scale)
        assert_close(o_lat[sl], ref_o, "bf16", f"{name} o_lat b={b}")
        assert np.max(np.abs(lse[sl] - ref_lse)) <= 1e-2, f"{name} lse b={b}"

    # the layer output against the explicit float64 chain, sampled sequences
    for i, b in enumerate(samples(p)):
        ref = oracle_sequence(p, b, explicit=(i == 0 and int(p.kv_len[b]) <= 16384))
        assert_close(out[b * n_q:(b + 1) * n_q], ref["out"], "bf16", f"{name} out b={b}")

    # appended cache rows (reading c13; reduced-precision rows within one code spacing, reading c21)
    check_rows = assert_fp8_rows_close if p.w.cache_fp8 else assert_append_c13
    if p.w.n_append:
        rows = L.cache_rows_at(np.repeat(np.arange(p.w.batch), n_q), p.q_pos)
        check_rows(rows, p.x_q, W["W_DKV"], W["W_KR"], p.q_pos, d.rope_base, f"{name} appended rows")
    if p.w.fill == "append":
        rng = np.random.default_rng(p.w.seed + 100)
        starts = np.concatenate([[0], np.cumsum(p.lens)[:-1]])
        pick = np.sort(rng.choice(int(p.lens.sum()), size=min(2048, int(p.lens.sum())), replace=False))
        seq = np.searchsorted(starts, pick, side="right") - 1
        pos = pick - starts[seq]
        got = L.cache_rows_at(seq, pos)
        check_rows(got, p.x_ctx[pick], W["W_DKV"], W["W_KR"], pos, d.rope_base, f"{name} built rows")
