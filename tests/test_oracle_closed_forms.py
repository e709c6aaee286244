"""Closed-form accounting the pages print, checked against ``oracle.accounting``.

* "Multi-Head Latent Attention: ..." Inference Economics table: MHA
  ``2 H d_h = 32,768``, GQA-8 ``2,048``, MLA ``d_c + d_R = 576``; 57x.
* "MLA Explained" Memory: 64x and 98.4 % for the latent alone; 503 GB vs
  7.9 GB at 128,000 tokens, 60 layers, bf16.
* "MLA, dim by dim" 4.1: 66.1M T vs 167.8M T (query side) and 22.0M T vs
  167.8M T (key side); 5.2: 32768/576 = 56.9x and the t coefficient
  ``4 h d_c + 2 h d_r + h = 278,656``.
* "From Vanilla Transformers to Modern LLMs -- Part 3", What goes into the
  KV cache: ``d_c = 4 d_h``, ``d_h^R = d_h / 2`` gives ``4.5 d_h``.
"""

import pytest

from oracle import accounting as acc

H, D_H, D_C, D_R = 128, 128, 512, 64
D_MODEL, D_QC = 5120, 1536


def test_cache_elements_per_token():
    assert acc.cache_elems_mha(H, D_H) == 32768
    assert acc.cache_elems_gqa(8, D_H) == 2048
    assert acc.cache_elems_mla(D_C, D_R) == 576
    assert round(acc.cache_elems_mha(H, D_H) / acc.cache_elems_mla(D_C, D_R), 1) == 56.9
    assert round(acc.cache_elems_mha(H, D_H) / acc.cache_elems_mla(D_C, D_R)) == 57
    assert acc.cache_elems_mha(H, D_H) // D_C == 64
    assert round(100 * (32768 - 512) / 32768, 1) == 98.4
    # "3.5x" versus 8-group GQA (2048 / 576 = 3.56, printed truncated)
    assert 3.5 <= acc.cache_elems_gqa(8, D_H) / acc.cache_elems_mla(D_C, D_R) < 3.6


def test_cache_in_units_of_head_dim():
    assert acc.cache_elems_mla(4 * D_H, D_H // 2) == 4.5 * D_H


def test_128k_context_bytes():
    T, L, bf16 = 128000, 60, 2
    mha = acc.cache_elems_mha(H, D_H) * L * T * bf16
    mla = D_C * L * T * bf16
    assert round(mha / 1e9) == 503
    assert round(mla / 1e9, 1) == 7.9


def test_contraction_flop_rule():
    # query side, "MLA, dim by dim" 4.1 (per token)
    factored = acc.contraction_flops([D_QC], D_MODEL) + acc.contraction_flops([H, D_H], D_QC)
    merged = acc.contraction_flops([H, D_H], D_MODEL)
    assert round(factored / 1e6, 1) == 66.1
    assert round(merged / 1e6, 1) == 167.8
    key_side = acc.contraction_flops([D_C], D_MODEL) + acc.contraction_flops([H, D_H], D_C)
    assert round(key_side / 1e6, 1) == 22.0


def test_decode_t_coefficient():
    assert acc.mla_decode_t_coefficient_with_rope(H, D_C, D_R) == 278656
    # the tensor-core part (no score add) is h fewer
    assert acc.decode_tensor_flops_per_token(H, D_C, D_R) == 278656 - H
    # without RoPE the cached-decode formula grows by 4 h d_c per token
    f1 = acc.mla_decode_flops_cached(D_MODEL, D_C, H, D_H, D_H, 1000)
    f2 = acc.mla_decode_flops_cached(D_MODEL, D_C, H, D_H, D_H, 1001)
    assert f2 - f1 == 4 * H * D_C


@pytest.mark.parametrize("t", [1, 64, 8192])
def test_decode_flops_terms(t):
    f = acc.mla_decode_flops_cached(D_MODEL, D_C, H, D_H, D_H, t)
    want = (2 * D_MODEL * D_C + 2 * H * D_MODEL * D_H + 2 * H * D_H * D_C + 4 * H * t * D_C
            + 2 * H * D_C * D_H + 2 * H * D_H * D_MODEL)
    assert f == want
