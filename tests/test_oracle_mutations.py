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
]


@pytest.mark.parametrize("name,bad,check", MUTATIONS, ids=[f"{m[0]}:{m[1].__name__}" for m in MUTATIONS])
def test_pin_catches_planted_mistake(monkeypatch, name, bad, check):
    monkeypatch.setattr(O, name, bad)
    with pytest.raises(AssertionError):
        check()
