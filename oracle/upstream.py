"""The projections that sit upstream of the decode hot path (fp64).

TEST INFRASTRUCTURE ONLY -- see the package docstring.

The hot path starts from an already-filled latent cache and already-projected
queries.  The tiny fp32 workload is specified by its hidden states and
weights instead, so the test harness uses these functions to turn them into
the path's inputs:

* down-projection ``c_t = W_DKV h_t`` ("Multi-Head Latent Attention: ...",
  MLA section; "From Vanilla Transformers to Modern LLMs -- Part 3" 2.b),
* RoPE key ``k_R = RoPE(W_KR h_t, t)`` and query ``q_R = RoPE(W_QR h_t, t)``
  ("MLA, dim by dim" 5.2; Part 3, 3.k and 3.l),
* content query ``q = W_Q h_t`` (no query compression, as in
  DeepSeek-V2-Lite: "MLA, dim by dim" section 3).

RoPE follows "MLA, dim by dim" section 3: adjacent coordinate pairs
``(2j, 2j+1)`` (0-based) are rotated by the angle ``t * theta_j`` with
``theta_j = base^(-2j/d)``, computed elementwise as
``x * cos + rotate_half(x) * sin`` where ``rotate_half`` maps the pair
``(x0, x1)`` to ``(-x1, x0)``.
"""

from __future__ import annotations

import numpy as np

from .mla import project


def rope_frequencies(d: int, base: float = 10000.0) -> np.ndarray:
    """``theta_j = base^(-2j/d)`` for ``j = 0 .. d/2 - 1``."""
    j = np.arange(d // 2, dtype=np.float64)
    return base ** (-2.0 * j / d)


def rotate_half(x: np.ndarray) -> np.ndarray:
    """Pairwise ``(x0, x1) -> (-x1, x0)`` on adjacent coordinates."""
    x = np.asarray(x, np.float64)
    out = np.empty_like(x)
    out[..., 0::2] = -x[..., 1::2]
    out[..., 1::2] = x[..., 0::2]
    return out


def rope(x: np.ndarray, position: float, theta: np.ndarray) -> np.ndarray:
    """Rotate the last axis of ``x`` for one position.

    Each adjacent pair ``j`` turns by ``position * theta[j]``.
    """
    x = np.asarray(x, np.float64)
    ang = np.repeat(position * np.asarray(theta, np.float64), 2)
    return x * np.cos(ang) + rotate_half(x) * np.sin(ang)


def down_project(W_DKV: np.ndarray, h: np.ndarray) -> np.ndarray:
    """``c = W_DKV h`` with ``W_DKV`` of shape ``[d_c, d]``."""
    return project(W_DKV, h)


def cache_row(h_t, W_DKV, W_KR, position, theta) -> np.ndarray:
    """The cache row of one token: ``[W_DKV h_t ; RoPE(W_KR h_t, position)]``.

    This is what the fused projection-and-append step writes ("Multi-Head
    Latent Attention: ...", MLA section: the latent and the shared RoPE key;
    "From Vanilla Transformers to Modern LLMs -- Part 3" 3.b, 3.k, 3.q: the
    key is cached already rotated at its own position).
    """
    c = down_project(W_DKV, h_t)
    k = rope(project(W_KR, h_t), position, theta)
    return np.concatenate([c, k])


def query_projection(h_t, W_Q, W_QR, H, d_h, d_r, position, theta):
    """The query of one token: ``q_nope[h] = (W_Q h_t)[h*d_h:(h+1)*d_h]`` and
    ``q_rope[h] = RoPE((W_QR h_t)[h*d_r:(h+1)*d_r], position)`` (no query
    compression; "Multi-Head Latent Attention: ...", the query and its
    per-head RoPE part; "From Vanilla Transformers to Modern LLMs -- Part 3"
    3.d, 3.l).  Returns ``(q_nope [H, d_h], q_rope [H, d_r])``."""
    q = project(W_Q, h_t).reshape(H, d_h)
    qr = project(W_QR, h_t)
    q_rope = np.stack([rope(qr[i * d_r:(i + 1) * d_r], position, theta) for i in range(H)])
    return q, q_rope


def tiny_workload_inputs(h, W_DKV, W_KR, W_Q, W_QR, H, d_h, d_r, base=10000.0):
    """Turn the tiny workload's hidden states and weights into decode inputs.

    ``h`` is ``[T, d]`` (token ``t`` at position ``t``).  The cache row of token
    ``j`` is ``[W_DKV h_j ; RoPE(W_KR h_j, j)]``; the query is taken from the
    last token: ``q_nope[h] = (W_Q h_T)[h*d_h:(h+1)*d_h]`` and
    ``q_rope[h] = RoPE((W_QR h_T)[h*d_r:(h+1)*d_r], T-1)``.

    Returns ``(cache_rows [T, d_c + d_r], q_nope [H, d_h], q_rope [H, d_r])``.
    """
    h = np.asarray(h, np.float64)
    T = h.shape[0]
    theta = rope_frequencies(d_r, base)
    c = down_project(W_DKV, h)  # [T, d_c]
    k_raw = project(W_KR, h)  # [T, d_r]
    k_r = np.stack([rope(k_raw[j], j, theta) for j in range(T)])
    q_all = project(W_Q, h[T - 1])  # [H*d_h]
    qr_all = project(W_QR, h[T - 1])  # [H*d_r]
    q_nope = q_all.reshape(H, d_h)
    q_rope = np.stack([rope(qr_all[i * d_r:(i + 1) * d_r], T - 1, theta)
                       for i in range(H)])
    return np.concatenate([c, k_r], axis=1), q_nope, q_rope
