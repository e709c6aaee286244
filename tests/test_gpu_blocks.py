"""GPU: decode over block ranges and the merge of the pieces.

``mla_decode_blocks`` over one range of logical cache blocks gives one
split-KV piece (``o_lat`` and ``lse`` over those keys alone); pieces over
ranges that partition the keys merge with ``mla_combine_pieces`` into the
whole decode.  This is the single-GPU form of splitting one long sequence
across GPUs (each call stands for one rank's range).  Checked against the
oracle's range-restricted decode and its log-sum-exp combine, at the
bf16 tolerances (max-abs 2e-2, mean-relative 5e-3), and against
``mla_decode`` itself.
"""

import numpy as np
import pytest
import torch

import synth
from harness import compact_sequence, compare, dims_for, f64, to_device
from oracle import mla as omla

pytestmark = pytest.mark.gpu

DS = dict(d_h=128, d_c=512, d_r=64)
BIG = 2**31 - 1


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mla_latent_kv_74_b300 as m
    return m


def _gpu(mla, inputs, ranges):
    """Append, absorb, then one mla_decode_blocks call per range, the merge of
    those pieces, and mla_decode; host copies of everything."""
    dev = to_device(inputs)
    d = dims_for(mla, inputs)
    B, Hq, H, _ = dev["q_nope"].shape
    ms = int(inputs["seqlens"].max())
    cache = dev["cache"].clone()
    mla.mla_append_cache(cache, inputs["num_blocks"], dev["block_table"], dev["seqlens"],
                         dev["c_kv_new"], dev["k_r_new"], d)
    q_lat = torch.empty(B, Hq, H, d.d_c, dtype=torch.bfloat16, device="cuda")
    mla.mla_absorb_query(dev["q_nope"], dev["W_UK"], q_lat, d)
    ws = mla.alloc_workspace(B, Hq, ms, d)
    P = len(ranges)
    o_p = torch.empty(P, B, Hq, H, d.d_c, dtype=torch.bfloat16, device="cuda")
    lse_p = torch.empty(P, B, Hq, H, dtype=torch.float32, device="cuda")
    for i, (first, end) in enumerate(ranges):
        mla.mla_decode_blocks(q_lat, dev["q_rope"], cache, inputs["num_blocks"],
                              dev["block_table"], dev["seqlens"], ms, first, end, d, o_p[i],
                              lse_p[i], ws)
    o_m = torch.empty(B, Hq, H, d.d_c, dtype=torch.bfloat16, device="cuda")
    lse_m = torch.empty(B, Hq, H, dtype=torch.float32, device="cuda")
    mla.mla_combine_pieces(o_p, lse_p, d, o_m, lse_m)
    o_full = torch.empty_like(o_m)
    lse_full = torch.empty_like(lse_m)
    mla.mla_decode(q_lat, dev["q_rope"], cache, inputs["num_blocks"], dev["block_table"],
                   dev["seqlens"], ms, d, o_full, lse_full, ws)
    torch.cuda.synchronize()
    return {
        "status": mla.mla_get_error(ws),
        "o_p": o_p.float().cpu().numpy(), "lse_p": lse_p.cpu().numpy(),
        "o_m": o_m.float().cpu().numpy(), "lse_m": lse_m.cpu().numpy(),
        "o_full": o_full.float().cpu().numpy(), "lse_full": lse_full.cpu().numpy(),
    }


def _oracle(inputs, ranges):
    """Per range: the oracle's decode restricted to the range (after the
    same append); and the whole decode."""
    B, Hq = inputs["q_nope"].shape[:2]
    W_UK, W_UV = f64(inputs["W_UK"]), f64(inputs["W_UV"])
    pieces = [([], []) for _ in ranges]
    full = ([], [])
    for b in range(B):
        cache, table = compact_sequence(inputs, b)
        sl = inputs["seqlens"][b:b + 1].numpy()
        cache = omla.append_to_cache(cache, table, sl, f64(inputs["c_kv_new"][b:b + 1]),
                                     f64(inputs["k_r_new"][b:b + 1]))
        qn, qr = f64(inputs["q_nope"][b:b + 1]), f64(inputs["q_rope"][b:b + 1])
        for i, (first, end) in enumerate(ranges):
            _, o, lse = omla.mla_decode_blocks(qn, qr, cache, table, sl, W_UK, W_UV, Hq,
                                               first, end)
            pieces[i][0].append(o)
            pieces[i][1].append(lse)
        _, o, lse = omla.mla_decode(qn, qr, cache, table, sl, W_UK, W_UV, Hq)
        full[0].append(o)
        full[1].append(lse)
    cat = np.concatenate
    return ([(cat(o), cat(l)) for o, l in pieces], (cat(full[0]), cat(full[1])))


CASES = {
    # name: (H, seqlens, Hq, ranges)
    # one long sequence cut into three ranks' ranges (each range itself cut
    # between several CTA pairs), plus short ones that end inside a range
    "long_three": (128, [5000, 70, 900], 1, [(0, 20), (20, 55), (55, BIG)]),
    # two query slots (causal), four ranges, one of them past every sequence
    "mtp_four": (128, [3000, 130, 64], 2, [(0, 1), (1, 2), (2, 40), (40, 100)]),
    # ranges of one block each at the start, then the rest
    "small_blocks": (128, [700, 65], 1, [(0, 1), (1, 2), (2, 3), (3, BIG)]),
    # few heads (one CTA per SM): two ranks' ranges, two query slots
    "few_heads": (16, [4000, 129, 1], 2, [(0, 30), (30, BIG)]),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_block_pieces_and_merge(mla, case):
    H, seqlens, Hq, ranges = CASES[case]
    inputs = synth.random_small(seed=21, H=H, seqlens=seqlens, Hq=Hq, **DS)
    res = _gpu(mla, inputs, ranges)
    assert res["status"] == 0
    pieces, (o_ref, lse_ref) = _oracle(inputs, ranges)
    for i, (o, lse) in enumerate(pieces):
        compare(res["o_p"][i], o, f"o_lat of range {ranges[i]}")
        compare(res["lse_p"][i], lse, f"lse of range {ranges[i]}")
    compare(res["o_m"], o_ref, "merged o_lat")
    compare(res["lse_m"], lse_ref, "merged lse")
    # the merge and the one-call decode agree within their bf16 roundings
    compare(res["o_m"], res["o_full"], "merged vs mla_decode o_lat")
    compare(res["lse_m"], res["lse_full"], "merged vs mla_decode lse")


@pytest.mark.parametrize("H", [128, 16])
def test_whole_range_is_the_decode(mla, H):
    """[0, INT_MAX) is the same computation as mla_decode: identical bytes."""
    inputs = synth.random_small(seed=22, H=H, seqlens=[2000, 1, 300], Hq=1, **DS)
    res = _gpu(mla, inputs, [(0, BIG)])
    assert res["status"] == 0
    assert np.array_equal(res["o_p"][0], res["o_full"])
    assert np.array_equal(res["lse_p"][0], res["lse_full"])


def test_empty_range_and_empty_pieces(mla):
    """A range past every sequence gives o = 0, lse = -inf; merged with the
    whole range it changes nothing; an empty range [k, k) likewise."""
    inputs = synth.random_small(seed=23, H=16, seqlens=[400, 129], Hq=1, **DS)
    res = _gpu(mla, inputs, [(0, BIG), (50, 60), (3, 3)])
    assert res["status"] == 0
    for i in (1, 2):
        assert np.all(res["o_p"][i] == 0) and np.all(np.isneginf(res["lse_p"][i]))
    compare(res["o_m"], res["o_full"], "merged with empty pieces")
    np.testing.assert_allclose(res["lse_m"], res["lse_full"], atol=1e-6)
