"""Closed-form cache sizes and FLOP counts (the pages' accounting).

TEST INFRASTRUCTURE ONLY -- see the package docstring.  ``bench.py`` keeps
its own copy of the per-token work formulas; tests check the two agree.

* Cache elements per token per layer: MHA ``2 H d_h``; MLA ``d_c + d_r``
  ("Multi-Head Latent Attention: ..." Inference Economics; "MLA Explained"
  Memory; "From Vanilla Transformers to Modern LLMs -- Part 3" 2.e, 3.q).
* Tensor-contraction FLOPs are ``2 * prod(output axes) * contracted axis``
  ("MLA, dim by dim" section 2).
* Cached MLA decode FLOPs ("MLA, dim by dim" 4.2, no RoPE, no Q compression):
  ``2 d d_c + 2 h d d_k + 2 h d_k d_c + 4 h t d_c + 2 h d_c d_v + 2 h d_v d``.
* With the decoupled RoPE branch the coefficient of ``t`` becomes
  ``4 h d_c + 2 h d_r + h`` ("MLA, dim by dim" 5.2, FLOPs supplement).
"""

from __future__ import annotations


def cache_elems_mha(H: int, d_h: int) -> int:
    return 2 * H * d_h


def cache_elems_gqa(groups: int, d_h: int) -> int:
    return 2 * groups * d_h


def cache_elems_mla(d_c: int, d_r: int) -> int:
    return d_c + d_r


def contraction_flops(output_axes, contracted: int) -> int:
    """``2 * prod(output axes) * k`` -- the GEMM counting convention."""
    n = 2 * contracted
    for a in output_axes:
        n *= a
    return n


def mla_decode_flops_cached(d, d_c, h, d_k, d_v, t):
    """Cached MLA decode FLOPs for one new token, no RoPE, no Q compression."""
    return (contraction_flops([d_c], d)            # x_t W_DKV
            + contraction_flops([h, d_k], d)       # x_t W_Q
            + contraction_flops([h, d_c], d_k)     # q W_UK^T (absorption)
            + contraction_flops([h, t], d_c)       # q_abs C^T
            + contraction_flops([h, d_c], t)       # p C
            + contraction_flops([h, d_v], d_c)     # o_c W_UV
            + contraction_flops([d], h * d_v))     # o W_o


def mla_decode_t_coefficient_with_rope(h, d_c, d_r):
    """Coefficient of ``t`` with the RoPE branch, counting the score add."""
    return 4 * h * d_c + 2 * h * d_r + h


def decode_tensor_flops_per_token(H, d_c, d_r):
    """Tensor-core FLOPs of the hot loop per visible token and query slot:
    ``QK^T`` over ``d_c + d_r`` plus ``P C`` over ``d_c`` (no score add)."""
    return contraction_flops([H], d_c + d_r) + contraction_flops([H, d_c], 1)


def prefill_attention_flops(T, H, d_qk, d_v, causal=True):
    """Tensor FLOPs of the prefill core attention of one ``T``-token sequence
    ("MLA, dim by dim" 4.1: ``S = Q K^T`` contracts ``d_qk``, ``O = P V``
    contracts the key axis into ``d_v``).  Dense, that is the pages'
    ``2 h T^2 (d_k + d_v)``; causal, only the ``T (T + 1) / 2`` visible
    (query, key) pairs count."""
    pairs = T * (T + 1) // 2 if causal else T * T
    return 2 * H * (d_qk + d_v) * pairs
