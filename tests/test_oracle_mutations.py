"""Planted mistakes in the oracle (on the CPU) must fail at least one pin.

Each mutation replaces one oracle function with a plausible wrong version
(a transposed operand, a dropped term, a wrong scale, an off-by-one) and
checks that the page pins in ``test_oracle_pins`` or the invariants catch
it.  This is what makes the pins meaningful: they are chosen so that every
step of the oracle is exercised by a number the pages print.
"""

import math

import numpy as np
import pytest

from oracle import mla, upstream
import test_oracle_pins as pins

ALL_PINS = (pins.check_prereq, pins.check_p5_upstream, pins.check_p5_content_path,
            pins.check_p5_norope_decode, pins.check_p5_full_decode,
            pins.check_projection_layouts)


def _some_pin_fails():
    for check in ALL_PINS:
        try:
            check()
        except AssertionError:
            return True
    return False


def _wrong_project(W, x):  # transposed operand
    W = np.asarray(W, np.float64)
    x = np.asarray(x, np.float64)
    if W.shape[0] == W.shape[1]:
        return x @ W
    return x @ W.T + 1e-3


def _keys_transposed(W_UK_h, c):
    return mla.project(np.asarray(W_UK_h).T, c)


def _values_from_keys_weight(W_UV_h, c):  # V rebuilt with the wrong matrix
    return mla.project(np.asarray(W_UV_h)[::-1], c)


def _scale_per_term(d_h, d_r):  # 1/sqrt(d_h) instead of the joint scale
    return 1.0 / math.sqrt(d_h)


def _visible_off_by_one(seqlen, Hq, slot):
    return max(0, int(seqlen) - int(Hq) + int(slot))


def _absorb_wrong_axis(q_nope, W_UK):
    return np.einsum("...ha,hca->...hc", np.asarray(q_nope, float),
                     np.asarray(W_UK, float).transpose(0, 2, 1)[:, ::-1])


def _rope_wrong_sign(x, position, theta):
    x = np.asarray(x, np.float64)
    ang = np.repeat(position * np.asarray(theta, np.float64), 2)
    return x * np.cos(ang) - upstream.rotate_half(x) * np.sin(ang)


def _attention_row_no_rope_term(q_nope, q_rope, rows, W_UK_h, W_UV_h, scale, d_c, K=None, V=None):
    return _ORIG_ROW(q_nope, np.zeros_like(np.asarray(q_rope, float)), rows, W_UK_h, W_UV_h,
                     scale, d_c, K=K, V=V)


def _attention_row_lse_without_max(q_nope, q_rope, rows, W_UK_h, W_UV_h, scale, d_c, K=None, V=None):
    r = _ORIG_ROW(q_nope, q_rope, rows, W_UK_h, W_UV_h, scale, d_c, K=K, V=V)
    if r["s"].size:
        r["lse"] = float(math.log(np.exp(r["s"] - r["s"].max()).sum()))
    return r


_ORIG_ROW = mla.attention_row


def _cache_row_unrotated(h_t, W_DKV, W_KR, position, theta):  # k_R cached before RoPE
    return np.concatenate([upstream.down_project(W_DKV, h_t), mla.project(W_KR, h_t)])


def _cache_row_rope_on_latent(h_t, W_DKV, W_KR, position, theta):  # rotates the wrong part
    c = upstream.down_project(W_DKV, h_t)
    k = mla.project(W_KR, h_t)
    return np.concatenate([upstream.rope(c, position, np.resize(theta, c.size // 2)), k])


def _query_rope_across_heads(h_t, W_Q, W_QR, H, d_h, d_r, position, theta):
    # all heads' RoPE parts rotated as one vector (frequencies of H*d_r)
    q = mla.project(W_Q, h_t).reshape(H, d_h)
    qr = mla.project(W_QR, h_t)
    th = upstream.rope_frequencies(H * d_r) * float(np.asarray(theta).ravel()[0])
    return q, upstream.rope(qr, position, th).reshape(H, d_r)


def _query_heads_interleaved(h_t, W_Q, W_QR, H, d_h, d_r, position, theta):
    # head h taken as every H-th coordinate instead of a contiguous slice
    q = mla.project(W_Q, h_t).reshape(d_h, H).T
    qr = mla.project(W_QR, h_t)
    return q, np.stack([upstream.rope(qr[i * d_r:(i + 1) * d_r], position, theta)
                        for i in range(H)])


def _output_projection_transposed(out, W_O):  # heads concatenated in the wrong order
    o = np.asarray(out, np.float64)
    return o.T.reshape(-1) @ np.asarray(W_O, np.float64)

MUTATIONS = {
    "project transposed": (mla, "project", _wrong_project),
    "keys use W_UK^T": (mla, "reconstruct_keys", _keys_transposed),
    "values use wrong W": (mla, "reconstruct_values", _values_from_keys_weight),
    "per-term scale": (mla, "default_scale", _scale_per_term),
    "visible length off by one": (mla, "visible_length", _visible_off_by_one),
    "absorb along wrong axis": (mla, "absorb_query", _absorb_wrong_axis),
    "RoPE wrong sign": (upstream, "rope", _rope_wrong_sign),
    "RoPE term dropped": (mla, "attention_row", _attention_row_no_rope_term),
    "lse drops the max": (mla, "attention_row", _attention_row_lse_without_max),
    "cache row k_R not rotated": (upstream, "cache_row", _cache_row_unrotated),
    "cache row rotates the latent": (upstream, "cache_row", _cache_row_rope_on_latent),
    "query RoPE across heads": (upstream, "query_projection", _query_rope_across_heads),
    "query heads interleaved": (upstream, "query_projection", _query_heads_interleaved),
    "W_O heads in wrong order": (mla, "output_projection", _output_projection_transposed),
}


def test_unmutated_oracle_passes_all_pins():
    assert not _some_pin_fails()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, monkeypatch):
    module, attr, fn = MUTATIONS[name]
    monkeypatch.setattr(module, attr, fn)
    assert _some_pin_fails(), f"mutation '{name}' slipped past every pin"
