"""The float64 oracle against brute force, a library routine, invariants,
special cases and the pages' printed numbers (CPU only)."""
import pytest

import pins


def test_page1_snippet_shapes():
    pins.check_page1_shapes()


@pytest.mark.parametrize("shape", [
    # tiny layer of the pages' numpy snippet (H=8, d=64, latent 64) with a 16-wide RoPE key, 10 tokens
    dict(d_model=512, H=8, qk_nope=64, d_rope=16, v_head=64, d_c=64, L=10, n_q=1),
    # smallest non-trivial case
    dict(d_model=6, H=2, qk_nope=3, d_rope=2, v_head=5, d_c=4, L=3, n_q=1),
    # two causal queries, unequal widths everywhere
    dict(d_model=10, H=3, qk_nope=4, d_rope=6, v_head=7, d_c=5, L=6, n_q=2),
])
def test_bruteforce_explicit(shape):
    pins.check_bruteforce(seed=1, **shape)


@pytest.mark.parametrize("shape", [
    dict(d_model=512, H=8, qk_nope=64, d_rope=16, v_head=64, d_c=64, L=10, n_q=1),
    dict(d_model=256, H=16, qk_nope=128, d_rope=64, v_head=128, d_c=512, L=200, n_q=2),
    dict(d_model=40, H=3, qk_nope=7, d_rope=4, v_head=9, d_c=11, L=33, n_q=2),
])
def test_absorbed_equals_explicit(shape):
    pins.check_absorbed_equals_explicit(seed=2, **shape)


@pytest.mark.parametrize("shape", [
    dict(d_model=512, H=8, qk_nope=64, d_rope=16, v_head=64, d_c=64, L=10, n_q=1),
    dict(d_model=256, H=128, qk_nope=128, d_rope=64, v_head=128, d_c=512, L=300, n_q=2),
])
def test_sdpa_library(shape):
    pins.check_sdpa(seed=3, **shape)


@pytest.mark.parametrize("shape", [
    # a whole prompt of 9 tokens, every token a query
    dict(d_model=40, H=3, qk_nope=7, d_rope=4, v_head=9, d_c=11, L=9, pos=list(range(9))),
    # scattered positions of a longer prompt, out of order, one of them the first token
    dict(d_model=64, H=4, qk_nope=16, d_rope=8, v_head=12, d_c=20, L=50, pos=[49, 0, 17, 31, 32, 8]),
])
def test_prefill_rows_against_sdpa(shape):
    pins.check_prefill_rows(seed=6, **shape)


def test_per_head_rope_keys():
    pins.check_per_head_rope()


def test_fp8_cache_format():
    pins.check_fp8_format()


def test_rope_properties():
    pins.check_rope_properties(16)
    pins.check_rope_properties(64)


def test_special_cases():
    pins.check_special_cases()


def test_merge_partials():
    pins.check_merge_partials()


def test_cache_closed_forms():
    pins.check_cache_closed_forms()


def test_round_bf16():
    pins.check_round_bf16()
