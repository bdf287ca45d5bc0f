"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins catch each one."""
import numpy as np
import pytest

import pins
from oracle import mla_oracle as O

TINY = dict(d_model=512, H=8, qk_nope=64, d_rope=16, v_head=64, d_c=64, L=10, n_q=1)
PAIR = dict(d_model=10, H=3, qk_nope=4, d_rope=6, v_head=7, d_c=5, L=6, n_q=2)


def _rope_wrong_direction(v, pos, base=10000.0):
    v = np.asarray(v, dtype=float)
    lead = v.shape[:-1]
    pos = np.broadcast_to(np.asarray(pos, dtype=float), lead)
    phi = O.rope_angles(pos.reshape(-1), v.shape[-1], base).reshape(*lead, v.shape[-1] // 2)
    out = np.empty_like(v)
    out[..., 0::2] = v[..., 0::2] * np.cos(phi) + v[..., 1::2] * np.sin(phi)
    out[..., 1::2] = -v[..., 0::2] * np.sin(phi) + v[..., 1::2] * np.cos(phi)
    return out


def _rope_half_split(v, pos, base=10000.0):
    v = np.asarray(v, dtype=float)
    d = v.shape[-1]
    perm = np.concatenate([np.arange(0, d, 2), np.arange(1, d, 2)])
    inv = np.argsort(perm)
    # rotate (i, i + d/2) pairs instead of interleaved ones
    return ORIG["apply_rope"](v[..., inv], pos, base)[..., perm]


ORIG = {name: getattr(O, name) for name in dir(O) if callable(getattr(O, name))}


def _attend_without_rope_term(q_nope, q_rope, c, k_r, W_UK, W_UV, kv_len, scale=None):
    return ORIG["attend_explicit"](q_nope, 0 * np.asarray(q_rope), c, k_r, W_UK, W_UV, kv_len, scale)


def _reconstruct_transposed(c, W_UK, W_UV, h):
    c = np.asarray(c, dtype=float)
    return c @ np.asarray(W_UK)[h], c @ np.asarray(W_UV)[h].T


def _attend_unscaled(q_nope, q_rope, c, k_r, W_UK, W_UV, kv_len, scale=None):
    return ORIG["attend_explicit"](q_nope, q_rope, c, k_r, W_UK, W_UV, kv_len, 1.0)


def _visible_off_by_one(kv_len, n_q, j):
    return max(0, int(kv_len) - (n_q - j))


def _absorb_transposed(q_nope, W_UK):
    return np.einsum("nhi,hci->nhc", np.asarray(q_nope, float), np.asarray(W_UK, float))


def _merge_unweighted(o_parts, lse_parts):
    o, lse = ORIG["merge_partials"](o_parts, lse_parts)
    return np.mean(np.asarray(o_parts), axis=0), lse


def _output_untransposed(o, W_O):
    o = np.asarray(o, float)
    return o.reshape(o.shape[0], -1) @ np.asarray(W_O, float)


def _query_without_rope(x, W_Q, W_QR, q_pos, n_heads, base=10000.0):
    return ORIG["project_query"](x, W_Q, W_QR, np.zeros_like(np.asarray(q_pos)), n_heads, base)


def _compress_unrotated(x, W_DKV, W_KR, pos, base=10000.0):
    return ORIG["compress"](x, W_DKV, W_KR, np.zeros_like(np.asarray(pos)), base)


def _prefill_window_off_by_one(q_nope, q_rope, pos, c, k_r, W_UK, W_UV, scale, store=None):
    # each query sees positions 0..pos-1 instead of 0..pos (its own token left out)
    pos = np.asarray(pos)
    o, lse = ORIG["attend_explicit_at"](q_nope, q_rope, np.maximum(pos - 1, 0), c, k_r, W_UK, W_UV, scale, store)
    return o, lse


def _prefill_first_head_key(q_nope, q_rope, pos, c, k_r, W_UK, W_UV, scale, store=None):
    # per-head keys read as one shared key (head 0's)
    k_r = np.asarray(k_r)
    if k_r.ndim == 3:
        k_r = k_r[:, 0]
    return ORIG["attend_explicit_at"](q_nope, q_rope, pos, c, k_r, W_UK, W_UV, scale, store)


def _e4m3_ties_away(x):
    x = np.asarray(x, dtype=float)
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    q = 2.0 ** (np.maximum(e, -6.0) - 3.0)
    return np.sign(x) * np.floor(a / q + 0.5) * q


def _e4m3_no_subnormal_clamp(x):
    x = np.asarray(x, dtype=float)
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    q = 2.0 ** (e - 3.0)                 # keeps 3 mantissa bits below 2^-6 as well
    return np.sign(x) * np.round(a / q) * q


def _e4m3_value_bias8(code):
    c = np.asarray(code, dtype=np.int64)
    sgn = np.where(c & 0x80, -1.0, 1.0)
    e, m = (c >> 3) & 0xF, c & 0x7
    val = np.where(e == 0, m / 8.0 * 2.0 ** -7, (1.0 + m / 8.0) * 2.0 ** (e - 8.0))
    return np.where((c & 0x7F) == 0x7F, np.nan, sgn * val)


def _scale_floor(c):
    m = np.max(np.abs(np.asarray(c, dtype=float)), axis=-1)
    return 2.0 ** np.floor(np.log2(np.where(m > 0, m, 448.0) / 448.0))


def _per_head_rope_flat(x, W_DKV, W_KR, pos, n_heads, base=10000.0):
    # one rotation over the whole H*d_rope row: frequencies do not restart in each head's key
    x = np.asarray(x, dtype=float)
    c = x @ np.asarray(W_DKV, dtype=float).T
    y = ORIG["apply_rope"](x @ np.asarray(W_KR, dtype=float).T, pos, base)
    return c, y.reshape(x.shape[0], n_heads, -1)


def _quantize_key_twice_scaled(c, k_r):
    codes, s, krs = ORIG["quantize_latent_fp8"](c, k_r)
    return codes, s, ORIG["round_bf16"](np.asarray(krs) / s[..., None])


MUTATIONS = [
    ("apply_rope", _rope_wrong_direction, lambda: pins.check_bruteforce(1, **TINY)),
    ("apply_rope", _rope_wrong_direction, lambda: pins.check_rope_properties(16)),
    ("apply_rope", _rope_half_split, lambda: pins.check_bruteforce(1, **TINY)),
    ("attend_explicit", _attend_without_rope_term, lambda: pins.check_bruteforce(1, **TINY)),
    ("attend_explicit", _attend_unscaled, lambda: pins.check_bruteforce(1, **TINY)),
    ("reconstruct_kv", _reconstruct_transposed, lambda: pins.check_bruteforce(1, **TINY)),
    ("visible", _visible_off_by_one, lambda: pins.check_bruteforce(1, **PAIR)),
    ("visible", _visible_off_by_one, lambda: pins.check_special_cases()),
    ("absorb_query", _absorb_transposed, lambda: pins.check_absorbed_equals_explicit(2, **TINY)),
    ("merge_partials", _merge_unweighted, lambda: pins.check_merge_partials()),
    ("output_project", _output_untransposed, lambda: pins.check_bruteforce(1, **TINY)),
    ("project_query", _query_without_rope, lambda: pins.check_bruteforce(1, **TINY)),
    ("compress", _compress_unrotated, lambda: pins.check_bruteforce(1, **TINY)),
    ("attend_explicit_at", _prefill_window_off_by_one,
     lambda: pins.check_prefill_rows(6, d_model=40, H=3, qk_nope=7, d_rope=4, v_head=9, d_c=11, L=9, pos=list(range(9)))),
    ("attend_explicit_at", _prefill_first_head_key, lambda: pins.check_per_head_rope()),
    ("round_e4m3", _e4m3_ties_away, lambda: pins.check_fp8_format()),
    ("round_e4m3", _e4m3_no_subnormal_clamp, lambda: pins.check_fp8_format()),
    ("e4m3_value", _e4m3_value_bias8, lambda: pins.check_fp8_format()),
    ("fp8_token_scale", _scale_floor, lambda: pins.check_fp8_format()),
    ("compress_per_head_rope", _per_head_rope_flat, lambda: pins.check_per_head_rope()),
    ("quantize_latent_fp8", _quantize_key_twice_scaled, lambda: pins.check_fp8_format()),
]


@pytest.mark.parametrize("name,bad,check", MUTATIONS, ids=[f"{m[0]}:{m[1].__name__}" for m in MUTATIONS])
def test_pin_catches_planted_mistake(monkeypatch, name, bad, check):
    monkeypatch.setattr(O, name, bad)
    with pytest.raises(AssertionError):
        check()
