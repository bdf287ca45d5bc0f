"""Prefill in the explicit form (per-head keys and values rebuilt from the cached latent, causal
attention per head) against the float64 oracle.

  * the attention call on drawn cache rows and queries, at prompt shapes that cover ragged query and
    key tiles, a chunk at the end of a longer prompt (query tiles straddling key tiles), one query,
    one cache block and a single token, with flat and sharp (x8) scores;
  * the whole chain from hidden states: append of the prompt, query projection, attention, output
    projection, against the pure float64 explicit chain;
  * the 4096-token prompt of the benchmark on sampled query rows;
  * two calls give identical bits; a bad block-table entry is flagged, not faulted.

Readings: the attention-stage oracle consumes the values the method stores (c15): the drawn bf16
cache rows and queries, and the rebuilt keys and values rounded to bf16 by the oracle's own rounding
(c20).  Tolerance: each query token's outputs within 2e-2 of that token's output RMS beyond half a
bf16 ulp (c12 applied per query token, c20); lse within 2e-2 in natural-log units."""
import numpy as np
import pytest
import torch

import mla_harness as Hn
import mla_inputs as I
from gpu_helpers import assert_close_rows
from oracle import mla_oracle as O

pytestmark = pytest.mark.gpu

SMALL = ["prefill_dsv2_L300_T300", "prefill_dsv2_L700_T200", "prefill_dsv2_L300_T1", "prefill_dsv2_L64_T64",
         "prefill_dsv2_L1_T1", "prefill_dsv2_L300_T300_rh"]
LSE_TOL = 2e-2


def oracle_rows(p: I.PrefillProblem, idx=None):
    d, W = p.dims, p.weights
    pos = p.q_pos if idx is None else p.q_pos[idx]
    q = (p.q if idx is None else p.q[idx]).astype(np.float64)
    rows = p.rows.astype(np.float64)
    k_r = rows[:, d.d_c:].reshape(rows.shape[0], d.n_heads, d.d_rope) if p.case.rope_per_head else rows[:, d.d_c:]
    return O.attend_explicit_at(q[..., :d.qk_nope], q[..., d.qk_nope:], pos, rows[:, :d.d_c], k_r,
                                W["W_UK"], W["W_UV"], O.softmax_scale(d.qk_nope, d.d_rope), store=O.round_bf16)


def run_attention(p: I.PrefillProblem):
    L = Hn.PrefillLayer(p)
    L.fill()
    L.attend()
    torch.cuda.synchronize()
    code, flags = L.status()
    assert code == 0, flags
    return L, L.o.float().cpu().numpy(), L.lse.cpu().numpy()


@pytest.mark.parametrize("sharp", [1.0, 8.0])
@pytest.mark.parametrize("name", SMALL)
def test_prefill_attention_matches_the_explicit_oracle(name, sharp):
    p = I.make_prefill(I.PREFILL_CASES[name], sharp=sharp)
    _, o, lse = run_attention(p)
    ref_o, ref_lse = oracle_rows(p)
    assert_close_rows(o, ref_o, f"{name} x{sharp:g} o")
    assert np.max(np.abs(lse - ref_lse)) <= LSE_TOL, f"{name} x{sharp:g} lse"


@pytest.mark.parametrize("name", ["prefill_dsv2_L333_T333_x", "prefill_dsv2_L333_T333_x_rh"])
def test_prefill_from_hidden_states_matches_the_float64_chain(name):
    c = I.PREFILL_CASES[name]
    p = I.make_prefill(c)
    d, W = p.dims, p.weights
    L = Hn.PrefillLayer(p)
    L.fill()
    L.run()
    torch.cuda.synchronize()
    code, flags = L.status()
    assert code == 0, flags
    xq = p.x[c.prompt - c.queries:]
    # the queries (stage check: the projection alone)
    q_nope, q_rope = O.project_query(xq, W["W_Q"], W["W_QR"], p.q_pos, d.n_heads, d.rope_base)
    q = L.q.float().cpu().numpy()
    assert_close_rows(q[..., :d.qk_nope], q_nope, "q_nope")
    assert_close_rows(q[..., d.qk_nope:], q_rope, "q_rope")
    # the layer output against the pure float64 explicit chain from the hidden states
    if c.rope_per_head:
        cc, k_r = O.compress_per_head_rope(p.x, W["W_DKV"], W["W_KR"], np.arange(c.prompt), d.n_heads, d.rope_base)
    else:
        cc, k_r = O.compress(p.x, W["W_DKV"], W["W_KR"], np.arange(c.prompt), d.rope_base)
    ref = O.decode_layer_explicit(xq, p.q_pos, [(cc, k_r)], W, d, c.queries, [c.prompt])
    assert_close_rows(L.out.float().cpu().numpy(), ref, "out")


def test_prefill_4096_token_prompt_on_sampled_rows():
    p = I.make_prefill(I.PREFILL_CASES["prefill_dsv2_L4096_T4096"])
    _, o, lse = run_attention(p)
    assert np.all(np.isfinite(o))
    T = p.case.queries
    rng = np.random.default_rng(p.case.seed + 1)
    idx = np.unique(np.concatenate([[0, 1, 127, 128, 2047, T - 129, T - 1], rng.choice(T, 17, replace=False)]))
    ref_o, ref_lse = oracle_rows(p, idx)
    assert_close_rows(o[idx], ref_o, "4096 sampled o")
    assert np.max(np.abs(lse[idx] - ref_lse)) <= LSE_TOL


def test_prefill_repeats_bit_for_bit():
    p = I.make_prefill(I.PREFILL_CASES["prefill_dsv2_L700_T200"])
    L, o1, lse1 = run_attention(p)
    L.attend()
    torch.cuda.synchronize()
    assert np.array_equal(L.o.view(torch.int16).cpu().numpy(), torch.from_numpy(o1).to(torch.bfloat16).view(torch.int16).numpy())
    assert np.array_equal(L.lse.cpu().numpy(), lse1)


def test_prefill_bad_block_entry_is_flagged_not_faulted():
    p = I.make_prefill(I.PREFILL_CASES["prefill_dsv2_L300_T300"])
    L = Hn.PrefillLayer(p)
    L.fill()
    L.block_table[p.case.seq, 2] = p.num_blocks + 5   # the prompt's third block points outside the pool
    L.attend()
    torch.cuda.synchronize()
    code, flags = L.status()
    assert code == 5 and flags & 1
    assert np.all(np.isfinite(L.o.float().cpu().numpy()))


def test_per_head_keys_are_refused_by_the_absorbed_decode():
    """The absorbed decode kernel shares one positional key across heads (an MMA operand); with per-head
    keys mla_decode_attention returns MLA_ERR_UNSUPPORTED and its workspace size is 0."""
    import ctypes
    import mla_latent_kv_81_b300 as M
    cfg = M.make_config(I.DSV2, "bf16", rope_per_head=True)
    assert M.mla_decode_workspace_bytes(cfg, 2, 1, 4) == 0
    cache = M.mla_paged_cache(0x2000, 8, 0x3000, 4, 2)
    fake = lambda n: ctypes.c_void_p(0x10000 * n)
    assert M.lib.mla_decode_attention(ctypes.byref(cfg), fake(1), ctypes.byref(cache), fake(2), 2, 1, fake(3), None,
                                      fake(4), 1 << 30, None) == 2
