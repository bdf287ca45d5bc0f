"""compress_append writes exactly the addressed rows of the paged cache, with the
values of the definition (GPU).  Bit-exactness criteria:
  (i)   placement: every row that is not addressed keeps its NaN sentinel bits;
  (ii)  one-hot weights and bf16-exact inputs at position 0: every stored value is exact;
  (iii) Gaussian inputs: every stored value is within one bf16 ulp (plus the
        fp32 accumulation error) of the float64 value, and equal to its
        round-to-nearest-even wherever the float64 value lies farther from a
        rounding midpoint than a wide estimate of the fp32 accumulation error
        (16 * 2u * sqrt(K) * ||w * x||_2, u = 2^-24)."""
import numpy as np
import pytest
import torch

import mla_harness as Hn
import mla_inputs as I
import mla_latent_kv_81_b300 as M
from oracle import mla_oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _layer(dims, dtype, lens, seed, n_append=0):
    w = I.Workload("pg", dims, dtype, len(lens), 1, 1, 1, n_append, seed, "append")
    return I.make_problem(w, lens=lens)


def _bf16_ulp(v):
    v = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(v, 1e-30)))
    return 2.0 ** (e - 7)


@pytest.mark.parametrize("dims,dtype", [(I.DSV2, "bf16"), (I.TINY, "f32")])
def test_append_placement_and_values(dims, dtype):
    lens = [3, 64, 130]
    p = _layer(dims, dtype, lens, 51)
    L = Hn.DeviceLayer(p)
    L.fill_by_append()
    torch.cuda.synchronize()
    code, _ = M.mla_get_device_status()
    assert code == 0
    flat = L.pool_rows().float().cpu().numpy()
    written = np.zeros(flat.shape[0], dtype=bool)
    start = 0
    for b, n in enumerate(lens):
        slots = I.paged_slots(p.block_table, b, np.arange(n), dims.block_size)
        written[slots] = True
        c, k_r = O.compress(p.x_ctx[start:start + n], p.weights["W_DKV"], p.weights["W_KR"], np.arange(n),
                            dims.rope_base)
        start += n
        ref = np.concatenate([c, k_r], axis=1)
        got = flat[slots].astype(np.float64)
        if dtype == "bf16":
            # (iii) within one ulp everywhere; exact where the fp32 accumulation cannot cross a midpoint
            # fp32 accumulation error estimate: 2u * sqrt(K) * ||w * x||_2, times a wide safety factor
            xs = p.x_ctx[start - n:start].astype(np.float64)
            u = 2.0 ** -23 * np.sqrt(dims.d_model) * 16
            acc_c = u * np.sqrt((xs * xs) @ (p.weights["W_DKV"].astype(np.float64) ** 2).T)
            y = xs @ p.weights["W_KR"].T.astype(np.float64)
            acc_y = u * np.sqrt((xs * xs) @ (p.weights["W_KR"].astype(np.float64) ** 2).T)
            # a rotated pair mixes both unrotated values; add the fp32 table and product roundings
            pair = acc_y[:, 0::2] + acc_y[:, 1::2] + 2.0 ** -20 * (np.abs(y[:, 0::2]) + np.abs(y[:, 1::2]))
            acc_bound = np.concatenate([acc_c, np.repeat(pair, 2, axis=1)], axis=1)
            rne = I.round_to_bf16(ref.astype(np.float32)).astype(np.float64)
            ulp = _bf16_ulp(ref)
            # within one ulp plus the accumulation estimate everywhere (near-zero values have tiny ulps)
            assert np.all(np.abs(got - ref) <= ulp + acc_bound)
            lo = np.floor(ref / ulp) * ulp
            dist_mid = np.abs(ref - (lo + ulp / 2))
            safe = dist_mid > acc_bound
            assert np.mean(safe) > 0.8, np.mean(safe)
            assert np.array_equal(got[safe], rne[safe])
        else:
            err = np.max(np.abs(got - ref) / np.maximum(np.abs(ref), np.sqrt(np.mean(ref ** 2))))
            assert err <= 1e-5
    # (i) every other row still holds NaN sentinels, bit for bit
    raw = L.pool_rows().view(torch.int16 if dtype == "bf16" else torch.int32).cpu().numpy()
    nan_bits = 0x7FC0 if dtype == "bf16" else 0x7FC00000
    untouched = raw[~written]
    assert np.all(untouched.astype(np.int64) & (0xFFFF if dtype == "bf16" else 0xFFFFFFFF) == nan_bits)


def test_append_one_hot_exact():
    """(ii) one-hot projection rows copy chosen inputs; RoPE at position 0 is the identity."""
    dims = I.DSV2
    p = _layer(dims, "bf16", [2], 52)
    rng = np.random.default_rng(52)
    W_DKV = np.zeros((dims.d_c, dims.d_model), dtype=np.float32)
    W_KR = np.zeros((dims.d_rope, dims.d_model), dtype=np.float32)
    src_c = rng.permutation(dims.d_model)[:dims.d_c]
    src_r = rng.permutation(dims.d_model)[:dims.d_rope]
    W_DKV[np.arange(dims.d_c), src_c] = 1.0
    W_KR[np.arange(dims.d_rope), src_r] = 1.0
    p.weights["W_DKV"], p.weights["W_KR"] = W_DKV, W_KR
    L = Hn.DeviceLayer(p)
    x = p.x_ctx[:1]
    M.mla_compress_append(L.cfg, Hn.to_dev(x, "bf16"), L.W["W_DKV"], L.W["W_KR"],
                          torch.zeros(1, dtype=torch.int32, device=DEV), torch.zeros(1, dtype=torch.int32, device=DEV),
                          L.rope, L.cache)
    torch.cuda.synchronize()
    row = L.pool_rows()[int(I.paged_slots(p.block_table, 0, [0], dims.block_size)[0])].cpu()
    expect = np.concatenate([x[0, src_c], x[0, src_r]])
    assert np.array_equal(row.view(torch.int16).numpy(), I.bf16_bits(expect).view(np.int16))
