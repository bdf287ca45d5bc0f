"""The C ABI on the host: the library loads, exports every symbol include/mla.h
declares, reports the per-token cache bytes of the closed form, and rejects bad
arguments before launching anything (no GPU needed)."""
import ctypes
import os
import re

import pytest

import mla_inputs as I
import mla_latent_kv_81_b300 as M
from oracle import mla_oracle as O

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "mla.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert len(names) >= 12
    for name in names:
        assert hasattr(M.lib, name), name
    assert set(M.EXPORTED) == set(names)


def test_status_strings():
    for code, name in M._binding.STATUS.items():
        assert M.mla_status_string(code) == name
    assert M.mla_status_string(99) == "MLA_ERR_UNKNOWN"


def test_cache_bytes_per_token_matches_closed_form():
    for dims, dtype, nbytes in ((I.DSV2, "bf16", 2), (I.TINY, "f32", 4)):
        cfg = M.make_config(dims, dtype)
        expect = O.cache_bytes(1, O.mla_cache_elems_per_token(dims.d_c, dims.d_rope), nbytes)
        assert M.mla_cache_bytes_per_token(cfg) == expect
    assert M.mla_cache_bytes_per_token(M.make_config(I.DSV2, "bf16")) == 1152
    assert M.mla_cache_bytes_per_token(M.make_config(I.TINY, "f32")) == 320
    # reduced-precision cache (reading c21): one byte per latent element, bf16 key, fp32 scale
    assert M.mla_cache_bytes_per_token(M.make_config(I.DSV2, "bf16", cache_fp8=True)) == 512 + 2 * 64 + 4
    assert M.mla_cache_bytes_per_token(M.make_config(I.TINY, "f32", cache_fp8=True)) == 0   # bf16 only
    bad = M.make_config(I.DSV2, "bf16")
    bad.cache_fp8 = 2
    assert M.mla_cache_bytes_per_token(bad) == 0
    # per-head positional keys: the row holds the latent and one key per head
    rh = M.make_config(I.DSV2, "bf16", rope_per_head=True)
    assert M.mla_cache_bytes_per_token(rh) == (512 + 128 * 64) * 2
    assert M.mla_decode_workspace_bytes(rh, 2, 1, 4) == 0          # absorbed decode: one shared key only
    assert M.mla_prefill_workspace_bytes(rh, 100) > M.mla_prefill_workspace_bytes(M.make_config(I.DSV2, "bf16"), 100)
    # the decode workspace of a reduced-precision cache also holds the expanded bf16 blocks
    f8 = M.make_config(I.DSV2, "bf16", cache_fp8=True)
    assert M.mla_decode_workspace_bytes(f8, 4, 1, 10) >= M.mla_decode_workspace_bytes(cfg := M.make_config(I.DSV2, "bf16"), 4, 1, 10) + 40 * 576 * 64 * 2


def test_invalid_config_is_rejected():
    cfg = M.make_config(I.TINY, "f32")
    cfg.d_rope = 15
    assert M.mla_cache_bytes_per_token(cfg) == 0
    cfg = M.make_config(I.TINY, "f32")
    cfg.dtype = 7
    assert M.mla_cache_bytes_per_token(cfg) == 0
    cfg = M.make_config(I.TINY, "f32")
    cfg.n_heads = 0
    assert M.mla_compress_workspace_bytes(cfg, 4) == 0


def test_workspace_sizes_cover_the_header_and_the_fp32_intermediates():
    for dims, dtype in ((I.TINY, "f32"), (I.DSV2, "bf16")):
        cfg = M.make_config(dims, dtype)
        assert M.mla_compress_workspace_bytes(cfg, 100) >= 256 + 100 * dims.row * 4
        H = dims.n_heads
        assert M.mla_absorb_workspace_bytes(cfg, 10) >= 256 + 10 * H * dims.qk_nope * 4
        assert M.mla_output_workspace_bytes(cfg, 10) >= 256 + 10 * H * dims.v_head * 2
        assert M.mla_decode_workspace_bytes(cfg, 4, 1, 1024) >= 256
        # every workspace, even for zero work, holds at least the status header
        assert M.mla_compress_workspace_bytes(cfg, 0) == 256
        assert M.mla_decode_workspace_bytes(cfg, 0, 1, 1) == 256


def test_bf16_shapes_outside_the_tensor_core_kernels_are_refused_on_the_host():
    """bf16 runs only on the tcgen05 kernels: a bf16 layer with 16 heads gets MLA_ERR_UNSUPPORTED from
    every entry point (after the pointer checks, before any device work) and a zero workspace size."""
    lib, byref = M.lib, ctypes.byref
    dims = I.Dims(d_model=256, n_heads=16, qk_nope=32, d_rope=32, v_head=48, d_c=256)
    cfg = M.make_config(dims, "bf16")
    UNS = 2
    assert M.mla_decode_workspace_bytes(cfg, 2, 1, 4) == 0
    assert M.mla_absorb_workspace_bytes(cfg, 2) == 0
    assert M.mla_output_workspace_bytes(cfg, 2) == 0
    assert M.mla_compress_workspace_bytes(cfg, 2) == 0
    rope = M.mla_rope_table(0x1000, 16)
    cache = M.mla_paged_cache(0x2000, 4, 0x3000, 2, 2)
    assert lib.mla_decode_attention(byref(cfg), _fake(1), byref(cache), _fake(2), 2, 1, _fake(3), None, _fake(4),
                                    1 << 30, None) == UNS
    assert lib.mla_absorb_query(byref(cfg), _fake(1), _fake(2), _fake(3), _fake(4), _fake(5), byref(rope), _fake(6), 2,
                                _fake(7), 1 << 30, None) == UNS
    assert lib.mla_output_project(byref(cfg), _fake(1), _fake(2), _fake(3), _fake(4), 2, _fake(6), 1 << 30,
                                  None) == UNS
    assert lib.mla_compress_append(byref(cfg), _fake(1), _fake(2), _fake(3), _fake(4), _fake(5), byref(rope),
                                   byref(cache), 2, _fake(6), 1 << 30, None) == UNS
    assert lib.mla_compress_append_noalloc(byref(cfg), _fake(1), _fake(2), _fake(3), _fake(4), _fake(5),
                                           byref(rope), byref(cache), 2, None) == UNS
    # the same shape in fp32 is supported (CUDA-core kernels)
    assert M.mla_decode_workspace_bytes(M.make_config(dims, "f32"), 2, 1, 4) >= 256


def test_reduced_precision_shapes_outside_its_kernels_are_refused_on_the_host():
    """The reduced-precision cache takes 64-token blocks, a latent in 64-column groups and at most 64
    positional columns: other shapes get MLA_ERR_UNSUPPORTED from every entry point and zero sizes."""
    lib, byref = M.lib, ctypes.byref
    UNS = 2
    rope = M.mla_rope_table(0x1000, 16)
    cache = M.mla_paged_cache(0x2000, 4, 0x3000, 2, 2)
    ok = M.make_config(I.DSV2, "bf16", cache_fp8=True)
    assert M.mla_cache_bytes_per_token(ok) == 512 + 2 * 64 + 4
    assert M.mla_compress_workspace_bytes(ok, 2) > 256
    for dims, bs in [(I.Dims(d_model=5120, n_heads=128, qk_nope=128, d_rope=128, v_head=128, d_c=512), 64),
                     (I.DSV2, 32)]:
        cfg = M.make_config(dims, "bf16", cache_fp8=True)
        cfg.block_size = bs
        assert M.mla_cache_bytes_per_token(cfg) == 0
        assert M.mla_compress_workspace_bytes(cfg, 2) == 0
        assert M.mla_decode_workspace_bytes(cfg, 2, 1, 4) == 0
        assert lib.mla_compress_append(byref(cfg), _fake(1), _fake(2), _fake(3), _fake(4), _fake(5), byref(rope),
                                       byref(cache), 2, _fake(6), 1 << 30, None) == UNS
        assert lib.mla_decode_attention(byref(cfg), _fake(1), byref(cache), _fake(2), 2, 1, _fake(3), None,
                                        _fake(4), 1 << 30, None) == UNS


def test_wait_timeout_selftest_rejects_long_limits_on_the_host():
    """The failure-detection self-check only accepts short limits (at most ~0.1 s of SM cycles) and a
    workspace holding the status header."""
    lib = M.lib
    assert lib.mla_selftest_wait_timeout(_fake(1), 256, 5000, None) == 1
    assert lib.mla_selftest_wait_timeout(_fake(1), 256, 400_000_000, None) == 1
    assert lib.mla_selftest_wait_timeout(None, 256, 2_000_000, None) == 6
    assert lib.mla_selftest_wait_timeout(_fake(1), 16, 2_000_000, None) == 6


def _fake(n):
    return ctypes.c_void_p(0x10000 * n)  # aligned, never dereferenced: validation fails first


def test_bad_arguments_fail_before_any_launch():
    lib = M.lib
    cfg = M.make_config(I.TINY, "f32")
    rope = M.mla_rope_table(0x1000, 16)
    cache = M.mla_paged_cache(0x2000, 4, 0x3000, 2, 1)
    INV, WS = 1, 6
    byref = ctypes.byref
    # null activation pointer
    assert lib.mla_compress_append(byref(cfg), None, _fake(1), _fake(2), _fake(3), _fake(4), byref(rope),
                                   byref(cache), 8, _fake(5), 1 << 20, None) == INV
    # misaligned weight pointer
    assert lib.mla_compress_append(byref(cfg), _fake(1), ctypes.c_void_p(0x10008), _fake(2), _fake(3), _fake(4),
                                   byref(rope), byref(cache), 8, _fake(5), 1 << 20, None) == INV
    # negative token count
    assert lib.mla_compress_append(byref(cfg), _fake(1), _fake(2), _fake(3), _fake(4), _fake(5), byref(rope),
                                   byref(cache), -1, _fake(6), 1 << 20, None) == INV
    # zero tokens is a no-op even with null pointers
    assert lib.mla_compress_append(byref(cfg), None, None, None, None, None, None, None, 0, None, 0, None) == 0
    # workspace too small, or null
    assert lib.mla_compress_append(byref(cfg), _fake(1), _fake(2), _fake(3), _fake(4), _fake(5), byref(rope),
                                   byref(cache), 8, _fake(6), 16, None) == WS
    assert lib.mla_compress_append(byref(cfg), _fake(1), _fake(2), _fake(3), _fake(4), _fake(5), byref(rope),
                                   byref(cache), 8, None, 1 << 20, None) == WS
    # misaligned workspace passed to the status read
    assert lib.mla_get_device_status(ctypes.c_void_p(0x10008), None, None) == INV
    # empty cache description
    bad_cache = M.mla_paged_cache(0x2000, 0, 0x3000, 2, 1)
    assert lib.mla_compress_append(byref(cfg), _fake(1), _fake(2), _fake(3), _fake(4), _fake(5), byref(rope),
                                   byref(bad_cache), 8, _fake(6), 1 << 20, None) == INV
    # decode: batch larger than the block table
    assert lib.mla_decode_attention(byref(cfg), _fake(1), byref(cache), _fake(2), 3, 1, _fake(3), None, _fake(4),
                                    1 << 30, None) == INV
    # decode: n_q = 0
    assert lib.mla_decode_attention(byref(cfg), _fake(1), byref(cache), _fake(2), 1, 0, _fake(3), None, _fake(4),
                                    1 << 30, None) == INV
    # decode: misaligned lse
    assert lib.mla_decode_attention(byref(cfg), _fake(1), byref(cache), _fake(2), 1, 1, _fake(3),
                                    ctypes.c_void_p(0x10004), _fake(4), 1 << 30, None) == INV
    # absorb / output: null output
    assert lib.mla_absorb_query(byref(cfg), _fake(1), _fake(2), _fake(3), _fake(4), _fake(5), byref(rope), None, 4,
                                _fake(6), 1 << 30, None) == INV
    assert lib.mla_output_project(byref(cfg), _fake(1), _fake(2), _fake(3), None, 4, _fake(6), 1 << 30, None) == INV
    # rope table: non-positive max_pos
    assert lib.mla_rope_table_create(byref(cfg), 10000.0, 0, _fake(1), None) == INV
    # unsupported: odd RoPE width
    odd = M.make_config(I.TINY, "f32")
    odd.d_rope = 15
    assert lib.mla_output_project(byref(odd), _fake(1), _fake(2), _fake(3), _fake(4), 4, _fake(6), 1 << 30,
                                  None) == 2


def test_prefill_entry_points_check_arguments_on_the_host():
    """The explicit-form calls: bf16 tensor-core shapes only, 1 <= T <= kv_len <= the sequence's
    blocks, seq inside the batch; all checked before any launch."""
    lib, byref = M.lib, ctypes.byref
    INV, UNS = 1, 2
    cfg = M.make_config(I.DSV2, "bf16")
    f32 = M.make_config(I.TINY, "f32")
    assert M.mla_prefill_workspace_bytes(cfg, 4096) >= 256 + 4096 * (576 + 2 * 128 * 128) * 2
    assert M.mla_prefill_workspace_bytes(cfg, 0) == 0
    assert M.mla_prefill_workspace_bytes(f32, 10) == 0
    assert M.mla_project_workspace_bytes(f32, 4) == 0
    assert M.mla_head_output_workspace_bytes(f32, 4) == 0
    assert M.mla_project_workspace_bytes(cfg, 0) == 256
    cache = M.mla_paged_cache(0x2000, 40, 0x3000, 4, 2)     # 4 blocks of 64 per sequence, 2 sequences
    args = lambda seq, kv, T: (byref(cfg), _fake(1), byref(cache), seq, kv, T, _fake(2), _fake(3), _fake(4), None,
                               _fake(5), 1 << 40, None)
    assert lib.mla_prefill_attention(*args(0, 100, 101)) == INV    # T > kv_len
    assert lib.mla_prefill_attention(*args(0, 100, 0)) == INV      # T = 0
    assert lib.mla_prefill_attention(*args(2, 100, 10)) == INV     # seq outside the batch
    assert lib.mla_prefill_attention(*args(0, 257, 10)) == INV     # more tokens than the sequence's blocks
    assert lib.mla_prefill_attention(byref(f32), _fake(1), byref(cache), 0, 8, 4, _fake(2), _fake(3), _fake(4),
                                     None, _fake(5), 1 << 40, None) == UNS
    rope = M.mla_rope_table(0x1000, 16)
    assert lib.mla_project_query(byref(f32), _fake(1), _fake(2), _fake(3), _fake(4), byref(rope), _fake(5), 4,
                                 _fake(6), 1 << 30, None) == UNS
    assert lib.mla_head_output_project(byref(f32), _fake(1), _fake(2), _fake(3), 4, _fake(6), 1 << 30, None) == UNS
    assert lib.mla_head_output_project(byref(cfg), None, _fake(2), _fake(3), 4, _fake(6), 1 << 30, None) == INV
