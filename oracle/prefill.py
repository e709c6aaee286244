"""MLA prefill in the standard (un-absorbed) order, fp64 (the oracle).

TEST INFRASTRUCTURE ONLY -- see the package docstring.

Sources (page title, section):

* "MLA, dim by dim" section 4.1 -- during prefill the keys and values are
  rebuilt from the latents first, ``K = C^KV W_UK`` and ``V = C^KV W_UV``,
  and only then do the two quadratic contractions ``S = Q K^T`` (over
  ``d_k``) and ``O = P V`` (over ``d_v``) run; absorbing the up-projections
  would move the quadratic terms onto ``d_c``.  The dense FLOP count of the
  core attention is ``2 h T^2 (d_k + d_v)``.
* "MLA Explained" -- training and prefill steps: compute the latent, expand
  K and V from it per head, then standard attention and a weighted sum of
  the values.
* "MLA, dim by dim" section 5.2 and "From Vanilla Transformers to Modern
  LLMs -- Part 3" 3.o -- the score adds the decoupled RoPE term (one rotated
  key per token, shared by the heads) and is scaled by ``1/sqrt(d_h + d_r)``.

Readings of points the pages leave open:

* The scores are the decode step's: content plus decoupled RoPE term, joint
  scale ``1/sqrt(d_h + d_r)`` (the "MLA Explained" sketch writes
  ``1/sqrt(d_h)`` without a RoPE term; the pages that treat the RoPE branch
  scale jointly).  So the last row of a prefill equals a decode of the same
  sequence.
* Prefill is causal: token ``t`` (0-based within its sequence) attends to
  tokens ``0 .. t``.
* Sequences are packed end to end (``cu_seqlens``, the prefix sums of their
  lengths); tokens never attend across a sequence boundary.
* ``lse`` is the natural log-sum-exp of the scaled scores, as in decode.

Layouts: ``q_nope [T, H, d_h]``, ``q_rope [T, H, d_r]`` (already rotated),
``c_kv [T, d_c]``, ``k_r [T, d_r]`` (already rotated), ``W_UK, W_UV
[H, d_h, d_c]``; outputs ``out [T, H, d_h]``, ``lse [T, H]``.
"""

from __future__ import annotations

import numpy as np


def up_project(W_h: np.ndarray, c: np.ndarray) -> np.ndarray:
    """Rebuild one head's keys or values from the latents: row ``j`` of the
    result is ``W_h c_j`` (``W_h`` is ``[d_h, d_c]``, ``c`` is ``[T, d_c]``)."""
    return np.asarray(c, np.float64) @ np.asarray(W_h, np.float64).T


def causal_softmax(s: np.ndarray):
    """Row-wise max-subtracted softmax of a ``[T, T]`` score matrix in which
    row ``t`` keeps only columns ``0 .. t``.  Returns ``(p, lse)``."""
    T = s.shape[0]
    visible = np.tril(np.ones((T, T), dtype=bool))
    masked = np.where(visible, s, -np.inf)
    m = masked.max(axis=1, keepdims=True)
    e = np.where(visible, np.exp(masked - m), 0.0)
    l = e.sum(axis=1, keepdims=True)
    return e / l, (m + np.log(l))[:, 0]


def prefill_sequence(q_nope, q_rope, c_kv, k_r, W_UK, W_UV, scale):
    """One sequence of ``T`` tokens, every head.

    Per head ``h``: ``K = c_kv W_UK[h]^T``, ``V = c_kv W_UV[h]^T``,
    ``S = (q_nope[:, h] K^T + q_rope[:, h] k_r^T) * scale``, causal softmax,
    ``out[:, h] = P V``.  Returns ``(out [T, H, d_h], lse [T, H])``.
    """
    q_nope = np.asarray(q_nope, np.float64)
    q_rope = np.asarray(q_rope, np.float64)
    c_kv = np.asarray(c_kv, np.float64)
    k_r = np.asarray(k_r, np.float64)
    T, H, d_h = q_nope.shape
    out = np.zeros((T, H, d_h))
    lse = np.zeros((T, H))
    if T == 0:
        return out, lse
    for h in range(H):
        K = up_project(W_UK[h], c_kv)  # [T, d_h]
        V = up_project(W_UV[h], c_kv)  # [T, d_h]
        s = (q_nope[:, h] @ K.T + q_rope[:, h] @ k_r.T) * scale
        p, lse[:, h] = causal_softmax(s)
        out[:, h] = p @ V
    return out, lse


def prefill(q_nope, q_rope, c_kv, k_r, W_UK, W_UV, cu_seqlens, scale):
    """Packed sequences: sequence ``b`` is tokens ``cu_seqlens[b] ..
    cu_seqlens[b+1] - 1`` of every input and output."""
    q_nope = np.asarray(q_nope, np.float64)
    T, H, d_h = q_nope.shape
    out = np.zeros((T, H, d_h))
    lse = np.zeros((T, H))
    for b in range(len(cu_seqlens) - 1):
        t0, t1 = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
        out[t0:t1], lse[t0:t1] = prefill_sequence(
            q_nope[t0:t1], q_rope[t0:t1], c_kv[t0:t1], k_r[t0:t1], W_UK, W_UV, scale)
    return out, lse


def prefill_row(q_nope_th, q_rope_th, c_kv, k_r, W_UK_h, W_UV_h, scale):
    """One (token, head) row: the query of token ``t = len(c_kv) - 1`` of
    head ``h`` against keys ``0 .. t`` (for sampled checks at large ``T``).
    Returns ``(out [d_h], lse)``."""
    K = up_project(W_UK_h, c_kv)
    V = up_project(W_UV_h, c_kv)
    s = (K @ np.asarray(q_nope_th, np.float64)
         + np.asarray(k_r, np.float64) @ np.asarray(q_rope_th, np.float64)) * scale
    m = s.max()
    e = np.exp(s - m)
    l = e.sum()
    return e @ V / l, float(m + np.log(l))
