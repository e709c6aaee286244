"""The seeded input generators: shapes, determinism and the value recipe
(activations N(0,1), up-projection weights N(0, 1/d_c), so scaled scores
have unit variance), and the packed prompts' prefix sums."""

import math

import numpy as np
import torch

import synth


def test_prefill_tensors_recipe():
    t = synth.prefill_tensors(seed=9, seqlens=[300, 0, 1200], H=8)
    T = 1500
    assert t["cu_seqlens"].tolist() == [0, 300, 300, 1500]
    assert t["cu_seqlens"].dtype == torch.int32
    assert tuple(t["q_nope"].shape) == (T, 8, 128) and tuple(t["q_rope"].shape) == (T, 8, 64)
    assert tuple(t["c_kv"].shape) == (T, 512) and tuple(t["k_r"].shape) == (T, 64)
    assert tuple(t["W_UK"].shape) == (8, 128, 512) and tuple(t["W_UV"].shape) == (8, 128, 512)
    for k in ("q_nope", "q_rope", "c_kv", "k_r", "W_UK", "W_UV"):
        assert t[k].dtype == torch.bfloat16, k
    for k in ("q_nope", "q_rope", "c_kv", "k_r"):
        x = t[k].double()
        assert abs(float(x.mean())) < 0.01 and abs(float(x.std()) - 1.0) < 0.01, k
    for k in ("W_UK", "W_UV"):
        assert abs(float(t[k].double().std()) * math.sqrt(512) - 1.0) < 0.01, k
    # rebuilt keys and their scaled scores have unit variance
    K = t["c_kv"].double() @ t["W_UK"][0].double().T
    assert abs(float(K.std()) - 1.0) < 0.03


def test_prefill_tensors_are_seeded():
    a = synth.prefill_tensors(seed=5, seqlens=[17, 3], H=2)
    b = synth.prefill_tensors(seed=5, seqlens=[17, 3], H=2)
    c = synth.prefill_tensors(seed=6, seqlens=[17, 3], H=2)
    for k in a:
        assert torch.equal(a[k], b[k]), k
    assert not torch.equal(a["q_nope"], c["q_nope"])


def test_paged_block_table_is_a_permutation():
    g = torch.Generator().manual_seed(3)
    seqlens = np.array([1, 64, 65, 200], dtype=np.int32)
    table, total = synth.paged_block_table(seqlens, 64, g)
    need = [1, 1, 2, 4]
    assert total == sum(need)
    used = np.concatenate([table[b, :n] for b, n in enumerate(need)])
    assert sorted(used.tolist()) == list(range(total))
    for b, n in enumerate(need):
        assert (table[b, n:] == -1).all()
