"""mla_compress_append_noalloc: the cache append for callers that cannot allocate device memory.

It keeps its scratch in a fixed array inside the library instead of a caller-provided workspace,
and runs the same kernels with the same split plan as the allocating mla_compress_append, so it
must write bit-identical cache rows."""
import ctypes

import numpy as np
import pytest
import torch

import mla_harness as Hn
import mla_inputs as I
import mla_latent_kv_81_b300 as M

SCRATCH_BYTES = 16 << 20
HEADER_BYTES = 256


def test_noalloc_scratch_covers_every_call_up_to_1024_tokens():
    """No GPU needed: the split plan is not monotone in T, so check every token count the documented
    promise covers, not only the largest."""
    cfg = M.make_config(I.DSV2, "bf16")
    for T in range(1, 1025):
        assert M.mla_compress_workspace_bytes(cfg, T) - HEADER_BYTES <= SCRATCH_BYTES, T


def test_noalloc_refuses_calls_larger_than_its_scratch():
    """No GPU needed: a call whose scratch exceeds the fixed 16 MiB is refused before any device work,
    after the same argument checks as mla_compress_append."""
    cfg = M.make_config(I.DSV2, "bf16")
    T = 65536
    assert M.mla_compress_workspace_bytes(cfg, T) - HEADER_BYTES > SCRATCH_BYTES
    rope = M.mla_rope_table(0x1000, 16)
    cache = M.mla_paged_cache(0x2000, 4, 0x3000, 2, 1)
    fake = [ctypes.c_void_p(0x10000 * i) for i in range(1, 6)]
    code = M.lib.mla_compress_append_noalloc(ctypes.byref(cfg), *fake, ctypes.byref(rope), ctypes.byref(cache), T,
                                             None)
    assert M.mla_status_string(code) == M.mla_status_string(6)   # MLA_ERR_WORKSPACE
    assert code == 6
    assert M.lib.mla_compress_append_noalloc(None, *fake, ctypes.byref(rope), ctypes.byref(cache), 4, None) == 1
    # a bad pointer is reported as such even when the call is also too large (same checks, same order)
    bad = [None] + fake[1:]
    assert M.lib.mla_compress_append_noalloc(ctypes.byref(cfg), *bad, ctypes.byref(rope), ctypes.byref(cache), T,
                                             None) == 1
    assert M.lib.mla_compress_append(ctypes.byref(cfg), *bad, ctypes.byref(rope), ctypes.byref(cache), T, None, 0,
                                     None) == 1


@pytest.mark.gpu
def test_noalloc_append_matches_the_allocating_append_on_two_calls():
    dims = I.DSV2
    lens = [130, 40, 300]
    w = I.Workload("noalloc", dims, "bf16", len(lens), 1, 1, 1, 0, 61, "direct")
    p = I.make_problem(w, lens=lens)
    ref = Hn.DeviceLayer(p)        # rows written by mla_compress_append (workspace from the caller)
    got = Hn.DeviceLayer(p)        # rows written by mla_compress_append_noalloc
    every = np.array([(b, q) for b, L in enumerate(lens) for q in range(L)], dtype=np.int32)
    rng = np.random.default_rng(61)
    for call, T in enumerate((37, 300)):
        # distinct (sequence, position) pairs, so no two tokens of a call write the same row
        pick = every[rng.choice(len(every), size=T, replace=False)]
        seq, pos = np.ascontiguousarray(pick[:, 0]), np.ascontiguousarray(pick[:, 1])
        x = Hn.to_dev(I.draw_hidden(rng, T, dims.d_model, "bf16"), "bf16")
        s_dev, p_dev = torch.from_numpy(seq).cuda(), torch.from_numpy(pos).cuda()
        ws = M.workspace(M.mla_compress_workspace_bytes(ref.cfg, T), "cuda")
        M.mla_compress_append(ref.cfg, x, ref.W["W_DKV"], ref.W["W_KR"], s_dev, p_dev, ref.rope, ref.cache, ws=ws)
        M.mla_compress_append_noalloc(got.cfg, x, got.W["W_DKV"], got.W["W_KR"], s_dev, p_dev, got.rope, got.cache)
        code, flags = M.mla_get_device_status(ws)
        assert code == 0, (M.mla_status_string(code), flags)
        code, flags = M.mla_get_device_status(None)   # the allocation-free call's flags
        assert code == 0, (M.mla_status_string(code), flags)
        # the same kernels with the same plan: the whole pool must be bit-identical, written rows and
        # untouched NaN sentinels alike
        assert torch.equal(ref.pool.view(torch.int16), got.pool.view(torch.int16)), f"call {call}"
        r_got = got.cache_rows_at(seq, pos)
        assert np.isfinite(r_got).all()
