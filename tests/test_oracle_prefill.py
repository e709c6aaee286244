"""Pins of the prefill oracle (``oracle.prefill``), and planted mistakes
that they must catch.

What fixes the prefill result independently of the code under test:

* every row of a prefill is one decode row: token ``t`` of head ``h``
  against the cached tokens ``0 .. t`` ("MLA, dim by dim" 4.1 and 4.2 run the
  same attention, once for all queries and once for the newest).  The decode
  row (``oracle.mla.attention_row``, written per row with explicit key and
  value reconstruction) is itself pinned to the pages' worked examples;
* a zero query scores every visible key equally, so the output is the
  running mean of the values, ``W_UV[h] mean(c_0 .. c_t)``, and
  ``lse = ln(t + 1)`` (closed form);
* a one-token sequence returns its own value ``W_UV[h] c_0`` and
  ``lse = s_00``;
* packed sequences never see each other's tokens;
* the causal attention FLOP count equals the number of visible
  (query, key) pairs, counted by enumeration, times ``2 H (d_qk + d_v)``;
  without the mask it is the pages' dense ``2 h T^2 (d_k + d_v)``.
"""

import math

import numpy as np
import pytest

from oracle import accounting, mla
from oracle import prefill as pf

# non-square, distinct sizes so a transposed or swapped operand cannot pass
H, D_H, D_C, D_R = 3, 5, 7, 4
SCALE = 1.0 / math.sqrt(D_H + D_R)


def _inputs(T, seed=0):
    rng = np.random.default_rng(seed)
    return {
        "q_nope": rng.standard_normal((T, H, D_H)),
        "q_rope": rng.standard_normal((T, H, D_R)),
        "c_kv": rng.standard_normal((T, D_C)),
        "k_r": rng.standard_normal((T, D_R)),
        "W_UK": rng.standard_normal((H, D_H, D_C)) / math.sqrt(D_C),
        "W_UV": rng.standard_normal((H, D_H, D_C)) / math.sqrt(D_C),
    }


def _run(x, cu=None):
    T = x["q_nope"].shape[0]
    cu = [0, T] if cu is None else cu
    return pf.prefill(x["q_nope"], x["q_rope"], x["c_kv"], x["k_r"], x["W_UK"], x["W_UV"],
                      cu, SCALE)


def check_rows_are_decode_rows():
    x = _inputs(9, seed=1)
    out, lse = _run(x)
    rows = np.concatenate([x["c_kv"], x["k_r"]], axis=1)
    for t in range(9):
        for h in range(H):
            r = mla.attention_row(x["q_nope"][t, h], x["q_rope"][t, h], rows[:t + 1],
                                  x["W_UK"][h], x["W_UV"][h], SCALE, D_C)
            np.testing.assert_allclose(out[t, h], r["out"], rtol=0, atol=1e-12)
            assert abs(lse[t, h] - r["lse"]) < 1e-12


def check_zero_query_running_mean():
    x = _inputs(6, seed=2)
    x["q_nope"][:] = 0.0
    x["q_rope"][:] = 0.0
    out, lse = _run(x)
    for t in range(6):
        mean_c = x["c_kv"][:t + 1].mean(axis=0)
        for h in range(H):
            np.testing.assert_allclose(out[t, h], x["W_UV"][h] @ mean_c, rtol=0, atol=1e-12)
            assert abs(lse[t, h] - math.log(t + 1)) < 1e-12


def check_single_token():
    x = _inputs(1, seed=3)
    out, lse = _run(x)
    for h in range(H):
        k = np.concatenate([x["W_UK"][h] @ x["c_kv"][0], x["k_r"][0]])
        q = np.concatenate([x["q_nope"][0, h], x["q_rope"][0, h]])
        np.testing.assert_allclose(out[0, h], x["W_UV"][h] @ x["c_kv"][0], rtol=0, atol=1e-12)
        assert abs(lse[0, h] - float(q @ k) * SCALE) < 1e-12


def check_packed_sequences_are_separate():
    x = _inputs(8, seed=4)
    out, lse = _run(x, cu=[0, 3, 8])
    for t0, t1 in ((0, 3), (3, 8)):
        part = {k: (v[t0:t1] if k not in ("W_UK", "W_UV") else v) for k, v in x.items()}
        o2, l2 = _run(part)
        np.testing.assert_allclose(out[t0:t1], o2, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[t0:t1], l2, rtol=0, atol=1e-12)
    # the first token of the second sequence sees only itself
    np.testing.assert_allclose(out[3], np.stack([x["W_UV"][h] @ x["c_kv"][3] for h in range(H)]),
                               rtol=0, atol=1e-12)


def check_prefill_row():
    x = _inputs(7, seed=5)
    out, lse = _run(x)
    for t in (0, 3, 6):
        for h in range(H):
            o, l = pf.prefill_row(x["q_nope"][t, h], x["q_rope"][t, h], x["c_kv"][:t + 1],
                                  x["k_r"][:t + 1], x["W_UK"][h], x["W_UV"][h], SCALE)
            np.testing.assert_allclose(o, out[t, h], rtol=0, atol=1e-12)
            assert abs(l - lse[t, h]) < 1e-12


def check_attention_flops():
    for T in (1, 2, 5, 64, 130):
        pairs = int(np.tril(np.ones((T, T), dtype=bool)).sum())  # enumerated
        per_pair = 2 * 128 * (192 + 128)
        assert accounting.prefill_attention_flops(T, 128, 192, 128) == pairs * per_pair
        # the pages' dense count: S = Q K^T over d_k, O = P V over d_v
        assert accounting.prefill_attention_flops(T, 128, 192, 128, causal=False) == (
            accounting.contraction_flops([128, T, T], 192)
            + accounting.contraction_flops([128, T, 128], T))


PINS = (check_rows_are_decode_rows, check_zero_query_running_mean, check_single_token,
        check_packed_sequences_are_separate, check_prefill_row)


@pytest.mark.parametrize("check", PINS + (check_attention_flops,), ids=lambda f: f.__name__)
def test_prefill_pin(check):
    check()


# ---- planted mistakes (CPU only) -------------------------------------------

_ORIG_SOFTMAX = pf.causal_softmax


def _mask_strict(s):  # token t misses itself
    T = s.shape[0]
    vis = np.tril(np.ones((T, T), dtype=bool), k=-1)
    vis[0, 0] = True
    masked = np.where(vis, s, -np.inf)
    m = masked.max(axis=1, keepdims=True)
    e = np.where(vis, np.exp(masked - m), 0.0)
    l = e.sum(axis=1, keepdims=True)
    return e / l, (m + np.log(l))[:, 0]


def _mask_transposed(s):  # attends to the future instead of the past
    p, lse = _ORIG_SOFTMAX(np.asarray(s)[::-1, ::-1])
    return p[::-1, ::-1], lse[::-1]


def _lse_without_max(s):
    p, lse = _ORIG_SOFTMAX(s)
    T = s.shape[0]
    vis = np.tril(np.ones((T, T), dtype=bool))
    m = np.where(vis, s, -np.inf).max(axis=1)
    return p, lse - m


def _up_wrong_columns(W_h, c):  # contracts only part of the latent
    W = np.asarray(W_h, np.float64)
    return np.asarray(c, np.float64)[:, :W.shape[0]] @ W[:, :W.shape[0]].T


def _sequence_without_rope(q_nope, q_rope, c_kv, k_r, W_UK, W_UV, scale):
    return _ORIG_SEQ(q_nope, np.zeros_like(np.asarray(q_rope, float)), c_kv, k_r, W_UK, W_UV,
                     scale)


def _sequence_values_from_keys(q_nope, q_rope, c_kv, k_r, W_UK, W_UV, scale):
    return _ORIG_SEQ(q_nope, q_rope, c_kv, k_r, W_UK, W_UK, scale)


def _prefill_ignores_boundaries(q_nope, q_rope, c_kv, k_r, W_UK, W_UV, cu_seqlens, scale):
    return _ORIG_SEQ(q_nope, q_rope, c_kv, k_r, W_UK, W_UV, scale)


_ORIG_SEQ = pf.prefill_sequence

MUTATIONS = {
    "mask_excludes_diagonal": ("causal_softmax", _mask_strict),
    "mask_transposed": ("causal_softmax", _mask_transposed),
    "lse_without_max": ("causal_softmax", _lse_without_max),
    "up_projection_wrong_columns": ("up_project", _up_wrong_columns),
    "rope_term_dropped": ("prefill_sequence", _sequence_without_rope),
    "values_from_keys_weight": ("prefill_sequence", _sequence_values_from_keys),
    "sequences_mixed": ("prefill", _prefill_ignores_boundaries),
}


def _some_pin_fails():
    for check in PINS:
        try:
            check()
        except AssertionError:
            return True
    return False


def test_unmutated_prefill_oracle_passes():
    assert not _some_pin_fails()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_prefill_mutation_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(pf, attr, fn)
    assert _some_pin_fails(), name
