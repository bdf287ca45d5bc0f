"""compress_append writes exactly the addressed rows of the paged cache, with the
values of the definition (GPU).  Bit-exactness criteria:
  (i)   placement: every row that is not addressed keeps its NaN sentinel bits;
  (ii)  one-hot weights and bf16-exact inputs at position 0: every stored value is exact;
  (iii) Gaussian inputs: every stored value is within one bf16 ulp (plus the
        fp32 accumulation error) of the float64 value, and equal to its
        round-to-nearest-even wherever the float64 value lies farther from a
        rounding midpoint than a wide estimate of the fp32 accumulation error
        (gpu_helpers.assert_append_c13)."""
import numpy as np
import pytest
import torch

import mla_harness as Hn
import mla_inputs as I
import mla_latent_kv_81_b300 as M
from gpu_helpers import assert_append_c13
from oracle import mla_oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _layer(dims, dtype, lens, seed, n_append=0):
    w = I.Workload("pg", dims, dtype, len(lens), 1, 1, 1, n_append, seed, "append")
    return I.make_problem(w, lens=lens)


@pytest.mark.parametrize("dims,dtype", [(I.DSV2, "bf16"), (I.TINY, "f32")])
def test_append_placement_and_values(dims, dtype):
    lens = [3, 64, 130]
    p = _layer(dims, dtype, lens, 51)
    L = Hn.DeviceLayer(p)
    L.fill_by_append()
    torch.cuda.synchronize()
    code, _ = L.status()
    assert code == 0
    written = np.zeros((p.num_blocks, dims.block_size), dtype=bool)
    start = 0
    for b, n in enumerate(lens):
        pos = np.arange(n)
        written[p.block_table[b, pos // dims.block_size], pos % dims.block_size] = True
        got = L.cache_rows_at(np.full(n, b), pos).astype(np.float64)
        x = p.x_ctx[start:start + n]
        start += n
        if dtype == "bf16":
            assert_append_c13(got, x, p.weights["W_DKV"], p.weights["W_KR"], pos, dims.rope_base, f"b={b}")
        else:
            c, k_r = O.compress(x, p.weights["W_DKV"], p.weights["W_KR"], pos, dims.rope_base)
            ref = np.concatenate([c, k_r], axis=1)
            err = np.max(np.abs(got - ref) / np.maximum(np.abs(ref), np.sqrt(np.mean(ref ** 2))))
            assert err <= 1e-5
    # (i) every other row still holds NaN sentinels, bit for bit
    nan_bits = 0x7FC0 if dtype == "bf16" else 0x7FC00000
    raw = L.pool_token_bits()   # [num_blocks, block_size, row] raw bit patterns
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
    row = L.cache_rows_at([0], [0])[0]
    expect = np.concatenate([x[0, src_c], x[0, src_r]])
    assert np.array_equal(I.bf16_bits(row).view(np.int16), I.bf16_bits(expect).view(np.int16))
