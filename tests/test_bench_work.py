"""The benchmark's algorithmic work counts agree with the oracle's closed
forms (``oracle.accounting``, pinned to the pages' printed numbers): the
decode's tensor FLOPs per visible (token, query slot) and the prefill's
rebuild and causal-attention FLOPs."""

import numpy as np

import bench
import synth
from oracle import accounting as acc


def test_decode_flops_match_the_accounting():
    w = synth.WORKLOADS["mtp"]
    seqlens = np.array([300, 1, 4096, 65], dtype=np.int64)
    flops, bytes_ = bench.decode_work(w, seqlens)
    visible = sum(max(0, int(s) - w.Hq + i + 1) for s in seqlens for i in range(w.Hq))
    assert bench.visible_tokens(seqlens, w.Hq) == visible
    assert flops == visible * acc.decode_tensor_flops_per_token(w.H, w.d_c, w.d_r)
    # the cache is read once per sequence, shared by heads and query slots
    assert bytes_ >= int(seqlens.sum()) * (w.d_c + w.d_r) * 2


def test_prefill_flops_match_the_accounting():
    seqlens = [4096, 7, 129, 1]
    kv, attn = bench.prefill_work(seqlens, 128)
    assert kv == acc.contraction_flops([sum(seqlens), 128, 2 * 128], 512)
    assert attn == sum(acc.prefill_attention_flops(n, 128, 128 + 64, 128) for n in seqlens)
