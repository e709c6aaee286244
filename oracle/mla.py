"""MLA decode, written out as its plain definition in fp64 (the oracle).

TEST INFRASTRUCTURE ONLY -- see the package docstring.

Sources (page title, section):

* "Multi-Head Latent Attention: Low-Rank KV Compression, Decoupled RoPE, and
  Matrix Absorption" -- MLA section: ``k_{s,i} = W_i^UK c_s``,
  ``v_{s,i} = W_i^UV c_s`` with ``W_i^UK, W_i^UV`` of shape ``d_h x d_c``.
  The library keeps that orientation: ``W_UK[h]`` is ``[d_h, d_c]``.
* "MLA, dim by dim" section 5.2 -- the score is the content term plus the
  decoupled RoPE term, scaled jointly by ``1/sqrt(d_k + d_r)``; the RoPE key
  is one vector per token shared by all heads and is cached already rotated.
* "From Vanilla Transformers to Modern LLMs -- Part 3" sections 3.e.1 (naive
  route: expand every cached latent into a key), 3.g (values), 3.o (combine
  content and position, scale 1/sqrt(d_h + d_h^R)), 3.p.
* "MLA Explained" -- decode steps: every cached latent is expanded to K and
  V, attention runs, the latent of the new token is appended.

The oracle deliberately takes the *un-absorbed* route: for every visible
cached token it rebuilds the per-head key ``K_j = W_UK[h] c_j`` and value
``V_j = W_UV[h] c_j`` and then runs a max-subtracted softmax.  Absorption is
an exact identity ("Mathematical Prerequisites for DeepSeek-V2" sections 6
and 7), so the absorbed GPU path must agree with this up to rounding.

Readings of points the pages leave open:

* ``seqlens[b]`` counts cached tokens *after* the ``Hq`` current tokens have
  been appended; query slot ``i`` of ``Hq`` sees positions
  ``0 .. seqlens[b] - Hq + i`` (causal between the query slots).
* A row with no visible token has ``o = 0`` and ``lse = -inf``.
* ``lse`` is the natural log-sum-exp of the scaled scores.
* Tensors are indexed ``[B, Hq, H, ...]``; the paged cache is
  ``[num_blocks, block_size, d_c + d_r]`` whose row holds ``[c_KV ; k_R]``.
"""

from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------------------
# building blocks ("Mathematical Prerequisites for DeepSeek-V2")
# ---------------------------------------------------------------------------


def project(W: np.ndarray, x: np.ndarray) -> np.ndarray:
    """Matrix-vector product ``y = W x`` (section 1), batched over leading
    axes of ``x``: ``x[..., n] -> y[..., m]`` for ``W`` of shape ``[m, n]``.
    """
    W = np.asarray(W, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    return x @ W.T


def dot(a: np.ndarray, b: np.ndarray) -> float:
    """Dot product ``a^T b`` (section 2)."""
    return float(np.dot(np.asarray(a, np.float64), np.asarray(b, np.float64)))


def concat_dot(a: np.ndarray, b: np.ndarray, c: np.ndarray, d: np.ndarray) -> float:
    """``[a; b]^T [c; d]`` computed on the concatenated vectors (section 9)."""
    return dot(np.concatenate([a, b]), np.concatenate([c, d]))


def bilinear_direct(a: np.ndarray, M: np.ndarray, b: np.ndarray) -> float:
    """``a^T (M b)``: apply ``M`` to ``b`` first (section 6, left side)."""
    return dot(a, project(M, b))


def bilinear_moved(a: np.ndarray, M: np.ndarray, b: np.ndarray) -> float:
    """``(M^T a)^T b``: move ``M`` onto ``a`` (section 6, right side)."""
    return dot(project(np.asarray(M, np.float64).T, a), b)


def weighted_sum_then_project(W: np.ndarray, alphas, xs) -> np.ndarray:
    """``W (sum_j alpha_j x_j)`` (section 7, left side)."""
    acc = sum(float(a) * np.asarray(x, np.float64) for a, x in zip(alphas, xs))
    return project(W, acc)


def project_then_weighted_sum(W: np.ndarray, alphas, xs) -> np.ndarray:
    """``sum_j alpha_j (W x_j)`` (section 7, right side)."""
    return sum(float(a) * project(W, x) for a, x in zip(alphas, xs))


def softmax(s: np.ndarray) -> np.ndarray:
    """Max-subtracted softmax of a 1-D score vector."""
    s = np.asarray(s, np.float64)
    e = np.exp(s - s.max())
    return e / e.sum()


# ---------------------------------------------------------------------------
# the paged latent cache
# ---------------------------------------------------------------------------


def visible_length(seqlen: int, Hq: int, slot: int) -> int:
    """Number of cached positions query slot ``slot`` of ``Hq`` may attend to.

    The current ``Hq`` tokens are appended before the step reads the cache
    ("MLA, dim by dim" 4.2: after appending, the step reads ``K_{<=t}``), and
    slot ``i`` sits at position ``seqlen - Hq + i``, so it sees that many
    positions plus one.
    """
    return max(0, int(seqlen) - int(Hq) + int(slot) + 1)


def gather_sequence(cache: np.ndarray, block_table_row: np.ndarray, n: int):
    """Logical rows ``0 .. n-1`` of one sequence, read through its block table.

    Position ``j`` lives in physical block ``block_table_row[j // bs]`` at slot
    ``j % bs``.  Returns the ``[n, d_c + d_r]`` rows as fp64.
    """
    bs = cache.shape[1]
    rows = [cache[int(block_table_row[j // bs]), j % bs] for j in range(n)]
    if n == 0:
        return np.zeros((0, cache.shape[2]), np.float64)
    return np.asarray(rows, dtype=np.float64)


def append_to_cache(cache, block_table, seqlens, c_kv, k_r):
    """Write the new tokens' ``[c_KV ; k_R]`` rows into a copy of the cache.

    New token ``i`` of sequence ``b`` goes to position
    ``seqlens[b] - n_new + i`` ("MLA Explained", decode step 5; "From Vanilla
    Transformers to Modern LLMs -- Part 3" 3.q: the rotated k_R is stored
    next to the latent).
    """
    out = np.array(cache, copy=True)
    B, n_new, d_c = c_kv.shape
    bs = cache.shape[1]
    for b in range(B):
        for i in range(n_new):
            pos = int(seqlens[b]) - n_new + i
            blk = int(block_table[b][pos // bs])
            out[blk, pos % bs, :d_c] = c_kv[b, i]
            out[blk, pos % bs, d_c:] = k_r[b, i]
    return out


# ---------------------------------------------------------------------------
# one attention row, un-absorbed
# ---------------------------------------------------------------------------


def reconstruct_keys(W_UK_h: np.ndarray, c: np.ndarray) -> np.ndarray:
    """``K_j = W_UK[h] c_j`` for every cached latent (the naive route)."""
    return project(W_UK_h, c)


def reconstruct_values(W_UV_h: np.ndarray, c: np.ndarray) -> np.ndarray:
    """``V_j = W_UV[h] c_j`` for every cached latent."""
    return project(W_UV_h, c)


def attention_row(q_nope, q_rope, rows, W_UK_h, W_UV_h, scale, d_c, K=None, V=None):
    """One (sequence, query slot, head) row of the decode step.

    ``rows`` are the visible cache rows ``[n, d_c + d_r]``.  ``K`` and ``V``
    may be passed in when they were already reconstructed for these rows
    (the two query slots of one sequence share them); otherwise they are
    rebuilt here.  Returns a dict with the scaled scores ``s``, probabilities
    ``p``, per-head output ``out`` (``d_h``), latent output ``o_lat`` (``d_c``)
    and ``lse``.
    """
    q_nope = np.asarray(q_nope, np.float64)
    q_rope = np.asarray(q_rope, np.float64)
    n = rows.shape[0]
    d_h = W_UK_h.shape[0]
    if n == 0:
        return {
            "s": np.zeros(0),
            "p": np.zeros(0),
            "out": np.zeros(d_h),
            "o_lat": np.zeros(d_c),
            "lse": -math.inf,
        }
    c = rows[:, :d_c]
    k_r = rows[:, d_c:]
    K = reconstruct_keys(W_UK_h, c) if K is None else K[:n]  # [n, d_h]
    V = reconstruct_values(W_UV_h, c) if V is None else V[:n]  # [n, d_h]
    # content score q^C . k^C_j plus positional score q^R . k^R_j, both taken
    # as one dot product of the concatenated vectors, then scaled jointly.
    s = (K @ q_nope + k_r @ q_rope) * scale
    m = s.max()
    e = np.exp(s - m)
    l = e.sum()
    p = e / l
    return {
        "s": s,
        "p": p,
        "out": p @ V,
        "o_lat": p @ c,
        "lse": float(m + math.log(l)),
    }


def default_scale(d_h: int, d_r: int) -> float:
    """``1 / sqrt(d_h + d_r)`` ("MLA, dim by dim" 5.2)."""
    return 1.0 / math.sqrt(d_h + d_r)


def mla_decode(q_nope, q_rope, cache, block_table, seqlens, W_UK, W_UV, Hq,
               scale=None, batch_indices=None, head_indices=None):
    """The whole decode step for the selected sequences.

    Shapes: ``q_nope [B, Hq, H, d_h]``, ``q_rope [B, Hq, H, d_r]``, ``cache
    [num_blocks, bs, d_c + d_r]``, ``block_table [B, max_blocks]``,
    ``seqlens [B]``, ``W_UK, W_UV [H, d_h, d_c]``.

    Returns ``out [nb, Hq, nh, d_h]``, ``o_lat [nb, Hq, nh, d_c]`` and
    ``lse [nb, Hq, nh]`` for the ``nb`` sequences in ``batch_indices`` and the
    ``nh`` heads in ``head_indices`` (all of them by default), in that order.
    """
    q_nope = np.asarray(q_nope, np.float64)
    q_rope = np.asarray(q_rope, np.float64)
    W_UK = np.asarray(W_UK, np.float64)
    W_UV = np.asarray(W_UV, np.float64)
    B, _, H, d_h = q_nope.shape
    d_c = W_UK.shape[2]
    if scale is None:
        scale = default_scale(d_h, q_rope.shape[3])
    if batch_indices is None:
        batch_indices = range(B)
    batch_indices = list(batch_indices)
    head_indices = list(range(H)) if head_indices is None else list(head_indices)
    nh = len(head_indices)
    out = np.zeros((len(batch_indices), Hq, nh, d_h))
    o_lat = np.zeros((len(batch_indices), Hq, nh, d_c))
    lse = np.full((len(batch_indices), Hq, nh), -math.inf)
    for ob, b in enumerate(batch_indices):
        n_max = visible_length(seqlens[b], Hq, Hq - 1)
        all_rows = gather_sequence(cache, block_table[b], n_max)
        for oh, h in enumerate(head_indices):
            # K_j and V_j of every visible position, rebuilt once per head and
            # shared by the query slots (slot i sees a prefix of them).
            K = reconstruct_keys(W_UK[h], all_rows[:, :d_c])
            V = reconstruct_values(W_UV[h], all_rows[:, :d_c])
            for i in range(Hq):
                n = visible_length(seqlens[b], Hq, i)
                r = attention_row(q_nope[b, i, h], q_rope[b, i, h], all_rows[:n],
                                  W_UK[h], W_UV[h], scale, d_c, K=K, V=V)
                out[ob, i, oh] = r["out"]
                o_lat[ob, i, oh] = r["o_lat"]
                lse[ob, i, oh] = r["lse"]
    return out, o_lat, lse


def mla_decode_blocks(q_nope, q_rope, cache, block_table, seqlens, W_UK, W_UV, Hq,
                      first_block, end_block, scale=None, batch_indices=None,
                      head_indices=None):
    """The decode step over the keys of logical blocks ``[first_block,
    end_block)`` only: position ``j`` takes part when ``first_block * bs <= j
    < end_block * bs`` and ``j`` is visible to the query slot.  The softmax
    is the same definition taken over that subset of the keys, so ``o_lat``
    and ``lse`` are one split-KV piece; a row with no key in the range has
    ``o = 0`` and ``lse = -inf``.  Shapes and returns as ``mla_decode``.
    (Not on the pages: it splits the key set the softmax of "From Vanilla
    Transformers to Modern LLMs -- Part 3" 2.a / 3.f runs over.)
    """
    q_nope = np.asarray(q_nope, np.float64)
    q_rope = np.asarray(q_rope, np.float64)
    W_UK = np.asarray(W_UK, np.float64)
    W_UV = np.asarray(W_UV, np.float64)
    B, _, H, d_h = q_nope.shape
    d_c = W_UK.shape[2]
    bs = cache.shape[1]
    if scale is None:
        scale = default_scale(d_h, q_rope.shape[3])
    batch_indices = list(range(B) if batch_indices is None else batch_indices)
    head_indices = list(range(H) if head_indices is None else head_indices)
    lo = max(0, int(first_block)) * bs
    hi = max(0, int(end_block)) * bs
    out = np.zeros((len(batch_indices), Hq, len(head_indices), d_h))
    o_lat = np.zeros((len(batch_indices), Hq, len(head_indices), d_c))
    lse = np.full((len(batch_indices), Hq, len(head_indices)), -math.inf)
    for ob, b in enumerate(batch_indices):
        n_max = visible_length(seqlens[b], Hq, Hq - 1)
        all_rows = gather_sequence(cache, block_table[b], n_max)
        for oh, h in enumerate(head_indices):
            for i in range(Hq):
                n = visible_length(seqlens[b], Hq, i)
                rows = all_rows[lo:min(n, hi)]
                r = attention_row(q_nope[b, i, h], q_rope[b, i, h], rows, W_UK[h], W_UV[h],
                                  scale, d_c)
                out[ob, i, oh] = r["out"]
                o_lat[ob, i, oh] = r["o_lat"]
                lse[ob, i, oh] = r["lse"]
    return out, o_lat, lse


def combine_pieces(o_pieces, lse_pieces):
    """Merge pieces computed over disjoint key sets: ``lse = ln sum_p
    exp(lse_p)`` and ``o = sum_p exp(lse_p - lse) o_p``.  With ``l_p`` the
    softmax denominator of piece ``p`` and ``m`` any shift, ``exp(lse_p) =
    l_p`` and the softmax over the union has denominator ``sum_p l_p``, so
    each piece's normalised output is re-weighted by its share of it.
    ``o_pieces [P, ..., d]``, ``lse_pieces [P, ...]``; a row with every
    ``lse_p = -inf`` has ``o = 0`` and ``lse = -inf``.
    """
    o_pieces = np.asarray(o_pieces, np.float64)
    lse_pieces = np.asarray(lse_pieces, np.float64)
    m = lse_pieces.max(axis=0)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    w = np.where(np.isfinite(lse_pieces), np.exp(lse_pieces - m_safe), 0.0)
    total = w.sum(axis=0)
    total_safe = np.where(empty, 1.0, total)
    o = (w[..., None] * o_pieces).sum(axis=0) / total_safe[..., None]
    o = np.where(empty[..., None], 0.0, o)
    lse = np.where(empty, -math.inf, m_safe + np.log(total_safe))
    return o, lse


# ---------------------------------------------------------------------------
# the absorbed quantities, by their definitions
# ---------------------------------------------------------------------------


def absorb_query(q_nope, W_UK):
    """``q_lat[.., h, :] = W_UK[h]^T q_nope[.., h, :]`` ("Multi-Head Latent
    Attention ..." Matrix Absorption; "From Vanilla Transformers to Modern
    LLMs -- Part 3" 3.e.2).  ``q_nope [..., H, d_h] -> [..., H, d_c]``.
    """
    q_nope = np.asarray(q_nope, np.float64)
    W_UK = np.asarray(W_UK, np.float64)
    return np.einsum("...ha,hac->...hc", q_nope, W_UK)


def out_proj(o_lat, W_UV):
    """``out[.., h, :] = W_UV[h] o_lat[.., h, :]`` (value up-projection applied
    once after the latent weighted sum; "From Vanilla Transformers to Modern
    LLMs -- Part 3" 3.g).  ``o_lat [..., H, d_c] -> [..., H, d_h]``.
    """
    o_lat = np.asarray(o_lat, np.float64)
    W_UV = np.asarray(W_UV, np.float64)
    return np.einsum("hac,...hc->...ha", W_UV, o_lat)


def absorbed_scores(q_lat_h, q_rope_h, rows, d_c, scale):
    """Scores taken directly against the cached latents:
    ``(q_lat . c_j + q_rope . k_R_j) * scale``.  Used only by the identity
    tests that check absorption against the un-absorbed route."""
    rows = np.asarray(rows, np.float64)
    return (rows[:, :d_c] @ np.asarray(q_lat_h, np.float64)
            + rows[:, d_c:] @ np.asarray(q_rope_h, np.float64)) * scale


def output_projection(out, W_O):
    """Concatenate the heads and apply ``W^O``: ``u = [o_1; ..; o_H] W^O``
    ("From Vanilla Transformers to Modern LLMs -- Part 3" 3.h; row-vector
    form, ``W_O`` of shape ``[H*d_h, d]``).  Only the worked-example test
    uses it: the library stops at the per-head ``out``."""
    return np.asarray(out, np.float64).reshape(-1) @ np.asarray(W_O, np.float64)
