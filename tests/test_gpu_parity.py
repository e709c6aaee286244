"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Sizes are chosen so the oracle finishes in seconds while still spanning
several 64-token tiles, ragged tails, empty rows, both query-slot counts and
both the tensor-core and CUDA-core shapes.  Tolerances: bf16 max-abs 2e-2 and
mean-relative 5e-3 (o_lat, lse, out, q_lat); fp32 1e-4.
"""

import json
import math
import os
import zlib

import numpy as np
import pytest
import torch

import synth
from harness import (compare, dims_for, f64, run_gpu_step, run_oracle_step, tiny_inputs,
                     to_device)
from oracle import mla as omla

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mla_latent_kv_74_b300 as m
    return m


def _check_step(res, inputs, dtype, batch_indices=None):
    out, o_lat, lse, q_lat = run_oracle_step(inputs, batch_indices)
    sel = list(range(inputs["q_nope"].shape[0])) if batch_indices is None else batch_indices
    compare(res["q_lat"], q_lat, "q_lat", dtype)
    compare(res["o_lat"][sel], o_lat, "o_lat", dtype)
    compare(res["lse"][sel], lse, "lse", dtype)
    compare(res["out"][sel], out, "out", dtype)
    assert res["status"] == 0


def test_tiny_fp32_workload(mla):
    inputs = tiny_inputs()
    res = run_gpu_step(mla, inputs)
    _check_step(res, inputs, "fp32")
    # append is a copy: the new row must be bit-exact
    assert torch.equal(res["cache"][0, 31], torch.cat([inputs["c_kv_new"][0, 0],
                                                       inputs["k_r_new"][0, 0]]))


def test_worked_example_fp32(mla):
    """The integer MLA step of "From Vanilla Transformers to Modern LLMs --
    Part 3" section 3 through the GPU (fp32), against the printed values."""
    g = json.load(open(os.path.join(GOLDEN, "towardsai_p3_worked_example.json")))
    pr = g["printed"]
    WUK = np.array(g["inputs"]["W_UK"]["value"], float)
    WUV = np.array(g["inputs"]["W_UV"]["value"], float)
    W_UK = np.ascontiguousarray(np.stack([WUK[:, h * 2:(h + 1) * 2].T for h in range(2)]))
    W_UV = np.ascontiguousarray(np.stack([WUV[:, h * 2:(h + 1) * 2].T for h in range(2)]))
    rows = np.concatenate([np.array(pr["latents"]["value"], float),
                           np.array(pr["k_R_cached"]["value"], float)], axis=1)
    # block size 2, blocks stored swapped; token 4 ("naimish") appended by the step
    cache = np.zeros((2, 2, 4))
    cache[1] = rows[0:2]
    cache[0, 0] = rows[2]
    f = lambda x: torch.tensor(np.asarray(x), dtype=torch.float32)
    inputs = {
        "cache": f(cache), "c_kv_new": f(rows[3:4, :2])[None], "k_r_new": f(rows[3:4, 2:])[None],
        "q_nope": f(pr["q4"]["value"]).reshape(1, 1, 2, 2),
        "q_rope": f([pr["q_R_head1"]["value"], pr["q_R_head2"]["value"]]).reshape(1, 1, 2, 2),
        "W_UK": f(W_UK), "W_UV": f(W_UV),
        "block_table": torch.tensor([[1, 0]], dtype=torch.int32),
        "seqlens": torch.tensor([4], dtype=torch.int32), "num_blocks": 2,
    }
    res = run_gpu_step(mla, inputs)
    _check_step(res, inputs, "fp32")
    np.testing.assert_allclose(res["o_lat"][0, 0, 0], pr["cbar_head1"]["value"], atol=1e-3)
    np.testing.assert_allclose(res["o_lat"][0, 0, 1], pr["cbar_head2"]["value"], atol=1e-3)
    np.testing.assert_allclose(res["out"][0, 0, 0], pr["o_head1"]["value"], atol=1e-3)
    np.testing.assert_allclose(res["out"][0, 0, 1], pr["o_head2"]["value"], atol=1e-3)
    np.testing.assert_allclose(res["q_lat"][0, 0, 0], pr["absorbed_query_head1"]["value"], atol=0)
    np.testing.assert_allclose(res["q_lat"][0, 0, 1], pr["absorbed_query_head2"]["value"], atol=0)


DS = dict(d_h=128, d_c=512, d_r=64)

CASES = {
    # name: (H, seqlens, Hq, extra)
    "h128_edges": (128, [1, 63, 64, 65, 300, 1000], 1, {}),
    "h128_mtp_causal": (128, [2, 5, 130, 777], 2, {}),
    "h128_short_rows": (128, [1, 3], 2, {}),  # seqlen < Hq leaves a row empty
    "h16_lite_like": (16, [100, 2049], 1, {}),
    # few heads, one CTA per SM: two causal slots, and H below 16
    "h16_mtp_causal": (16, [2, 5, 130, 777], 2, {}),
    "h16_short_rows": (16, [1, 3, 70], 2, {}),  # seqlen < Hq leaves a row empty
    "h8_few_heads": (8, [1, 64, 65, 3000], 1, {}),
    "h64_odd_heads": (64, [129, 7], 1, {}),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_bf16_deepseek_dims(mla, name):
    H, seqlens, Hq, _ = CASES[name]
    inputs = synth.random_small(seed=zlib.crc32(name.encode()) % 1000, H=H, seqlens=seqlens, Hq=Hq, **DS)
    res = run_gpu_step(mla, inputs)
    _check_step(res, inputs, "bf16")


@pytest.mark.parametrize("H", [8, 32])
def test_single_sequence_few_rows(mla, H):
    """One sequence, one slot: fewer query rows in all (H) than the query
    copy's box (16 rows with few heads, 64 in the pair kernel); the rows past
    the tensor read as zero."""
    inputs = synth.random_small(seed=15, H=H, seqlens=[300], Hq=1, **DS)
    res = run_gpu_step(mla, inputs)
    assert res["status"] == 0
    _check_step(res, inputs, "bf16")


@pytest.mark.parametrize("shape", [
    dict(H=3, d_h=40, d_c=72, d_r=16, bs=16, dtype=torch.bfloat16),
    dict(H=8, d_h=32, d_c=64, d_r=32, bs=32, dtype=torch.float32),
    dict(H=5, d_h=16, d_c=24, d_r=0, bs=8, dtype=torch.float32),
])
def test_other_shapes(mla, shape):
    dt = shape.pop("dtype")
    bs = shape.pop("bs")
    inputs = synth.random_small(seed=11, seqlens=[1, 17, 40, 100], Hq=2, block_size=bs,
                                dtype=dt, **shape)
    res = run_gpu_step(mla, inputs)
    _check_step(res, inputs, "bf16" if dt == torch.bfloat16 else "fp32")


def test_append_bit_exact(mla):
    inputs = synth.random_small(seed=5, H=4, seqlens=[3, 64, 65, 200], Hq=2, **DS)
    res = run_gpu_step(mla, inputs)
    bt = inputs["block_table"].numpy()
    want = omla.append_to_cache(inputs["cache"].float().numpy(), bt, inputs["seqlens"].numpy(),
                                inputs["c_kv_new"].float().numpy(),
                                inputs["k_r_new"].float().numpy())
    assert np.array_equal(res["cache"].float().numpy(), want)


def test_out_proj_alone(mla):
    """out_proj on a synthesised o_lat (not the decode's), against the oracle."""
    g = torch.Generator().manual_seed(21)
    for H, rows in ((128, 64), (16, 5), (128, 256)):
        o_lat = torch.randn(rows, 1, H, 512, generator=g).mul_(0.05).to(torch.bfloat16)
        W_UV = torch.randn(H, 128, 512, generator=g).div_(math.sqrt(512)).to(torch.bfloat16)
        d = mla.Dims(H=H, d_h=128, d_c=512, d_r=64, block_size=64, dtype=torch.bfloat16)
        out = torch.empty(rows, 1, H, 128, dtype=torch.bfloat16, device="cuda")
        mla.mla_out_proj(o_lat.cuda(), W_UV.cuda(), out, d)
        want = omla.out_proj(f64(o_lat), f64(W_UV))
        compare(out.float().cpu().numpy(), want, f"out_proj H={H} rows={rows}")


def test_absorb_alone_many_rows(mla):
    g = torch.Generator().manual_seed(22)
    for H, rows in ((128, 300), (16, 1)):
        q = torch.randn(rows, 1, H, 128, generator=g).to(torch.bfloat16)
        W = torch.randn(H, 128, 512, generator=g).div_(math.sqrt(512)).to(torch.bfloat16)
        d = mla.Dims(H=H, d_h=128, d_c=512, d_r=64, block_size=64, dtype=torch.bfloat16)
        q_lat = torch.empty(rows, 1, H, 512, dtype=torch.bfloat16, device="cuda")
        mla.mla_absorb_query(q.cuda(), W.cuda(), q_lat, d)
        compare(q_lat.float().cpu().numpy(), omla.absorb_query(f64(q), f64(W)),
                f"absorb H={H} rows={rows}")


def test_block_table_permutation_invariance(mla):
    """Moving the physical blocks (and the table with them) changes nothing,
    bit for bit."""
    inputs = synth.random_small(seed=8, H=128, seqlens=[200, 65, 129], Hq=1, **DS)
    ref = run_gpu_step(mla, inputs)
    nb = inputs["num_blocks"]
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(3))
    moved = dict(inputs)
    cache = torch.empty_like(inputs["cache"])
    cache[perm] = inputs["cache"]
    moved["cache"] = cache
    bt = inputs["block_table"].clone()
    m = bt >= 0
    bt[m] = perm[bt[m].long()].to(torch.int32)
    moved["block_table"] = bt
    got = run_gpu_step(mla, moved)
    for k in ("o_lat", "lse", "out"):
        assert np.array_equal(got[k], ref[k]), k


def _pieces(seqlens, Hq, npairs, item_cost=6, tile=64):
    """How many split pieces each (sequence, slot) item is cut into by the
    tensor-core decode's plan: items laid out slot by slot, each preceded by
    ``item_cost`` start-up units; with several slots (and at least as many
    pairs as slots) each slot's items are cut into equal ranges over its own
    share of the pairs, else all items over all pairs.  Used to show which
    piece counts a sweep covers."""
    groups = Hq if (Hq > 1 and npairs >= Hq) else 1
    per_group = npairs // groups
    slots = [list(range(Hq))] if groups == 1 else [[i] for i in range(Hq)]
    pieces = []
    for slot_set in slots:
        units, spans = 0, []
        for i in slot_set:
            for n_seq in seqlens:
                nt = -(-max(0, n_seq - Hq + i + 1) // tile)
                if nt:
                    spans.append((units + item_cost, units + item_cost + nt))
                    units += item_cost + nt
        per = -(-units // per_group)
        pieces += [(e - 1) // per - s // per + 1 for s, e in spans]
    return pieces


SPLIT_CASES = {
    # name: (H, seqlens, Hq, split counts swept, start-up units per item)
    "hq1": (128, [4000, 300, 64, 1, 900, 2500], 1, (1, 3, 7, 74), 6),
    "hq2": (128, [5000, 70, 5, 130], 2, (1, 3, 7, 74), 6),
    # few heads: one CTA per SM takes the place of a pair, up to 148 of them
    "h16": (16, [4000, 300, 64, 1, 900, 2500], 1, (1, 5, 7, 148), 2),
}


@pytest.mark.parametrize("case", sorted(SPLIT_CASES))
def test_split_invariance(mla, case):
    """The result does not depend on how the items are cut between CTA pairs
    (or, with few heads, CTAs): the split count of the plan is swept from 1
    to every pair (CTA), which cuts the longest item into 1, 2 or more, 3 or
    more and twenty to sixty pieces; every sweep point matches the oracle,
    and the points match one another within the rounding of the fp32
    partials."""
    H, seqlens, Hq, sweep, cost = SPLIT_CASES[case]
    inputs = synth.random_small(seed=9, H=H, seqlens=seqlens, Hq=Hq, **DS)
    out, o_lat, lse, _ = run_oracle_step(inputs)
    results = {}
    covered = set()
    try:
        for npairs in sweep:
            mla.mla_debug_set_decode_pairs(npairs)
            covered.add(max(_pieces(seqlens, Hq, npairs, item_cost=cost)))
            res = run_gpu_step(mla, inputs)
            assert res["status"] == 0
            compare(res["o_lat"], o_lat, f"o_lat pairs={npairs}")
            compare(res["lse"], lse, f"lse pairs={npairs}")
            compare(res["out"], out, f"out pairs={npairs}")
            results[npairs] = res
    finally:
        mla.mla_debug_set_decode_pairs(0)
    assert {1, 3}.issubset(covered) and max(covered) >= 10, covered
    ref = results[1]
    for npairs, res in results.items():
        for k in ("o_lat", "lse", "out"):
            compare(res[k], ref[k], f"{k} pairs={npairs} vs 1")


def test_deterministic(mla):
    inputs = synth.random_small(seed=10, H=128, seqlens=[700, 64], Hq=2, **DS)
    a = run_gpu_step(mla, inputs)
    b = run_gpu_step(mla, inputs)
    for k in ("o_lat", "lse", "out", "q_lat"):
        assert np.array_equal(a[k], b[k]), k


def test_few_heads_workspace_reuse(mla):
    """One workspace reused for several few-heads calls (one CTA per SM),
    with the split count changed between them, gives the same bytes for the
    same split every time, and every call matches the oracle."""
    inputs = synth.random_small(seed=14, H=16, seqlens=[1500, 65, 1, 700], Hq=1, **DS)
    dev = to_device(inputs)
    d = dims_for(mla, inputs)
    B, Hq, H, _ = dev["q_nope"].shape
    ms = int(inputs["seqlens"].max())
    q_lat = torch.empty(B, Hq, H, d.d_c, dtype=torch.bfloat16, device="cuda")
    mla.mla_absorb_query(dev["q_nope"], dev["W_UK"], q_lat, d)
    ws = mla.alloc_workspace(B, Hq, ms, d)
    outs = []
    try:
        for npairs in (0, 9, 0, 0):
            mla.mla_debug_set_decode_pairs(npairs)
            o = torch.empty(B, Hq, H, d.d_c, dtype=torch.bfloat16, device="cuda")
            lse = torch.empty(B, Hq, H, dtype=torch.float32, device="cuda")
            mla.mla_decode(q_lat, dev["q_rope"], dev["cache"], inputs["num_blocks"],
                           dev["block_table"], dev["seqlens"], ms, d, o, lse, ws)
            assert mla.mla_get_error(ws) == 0
            outs.append((o.float().cpu().numpy(), lse.cpu().numpy()))
    finally:
        mla.mla_debug_set_decode_pairs(0)
    for k in (2, 3):
        assert np.array_equal(outs[k][0], outs[0][0]) and np.array_equal(outs[k][1], outs[0][1])
    compare(outs[1][0], outs[0][0], "o_lat, 9 CTAs vs all")
    compare(outs[1][1], outs[0][1], "lse, 9 CTAs vs all")
    _, o_ref, lse_ref = omla.mla_decode(f64(inputs["q_nope"]), f64(inputs["q_rope"]),
                                        f64(inputs["cache"]), inputs["block_table"].numpy(),
                                        inputs["seqlens"].numpy(), f64(inputs["W_UK"]),
                                        f64(inputs["W_UV"]), Hq)
    compare(outs[0][0], o_ref, "o_lat")
    compare(outs[0][1], lse_ref, "lse")


@pytest.mark.parametrize("H", [128, 16])
def test_bad_block_index_reported(mla, H):
    """A table entry outside [0, num_blocks) is flagged on the device; that
    sequence's rows come back as 0 / -inf and the others are untouched."""
    inputs = synth.random_small(seed=12, H=H, seqlens=[130, 200], Hq=1, **DS)
    good = run_gpu_step(mla, inputs)
    bad = dict(inputs)
    bt = inputs["block_table"].clone()
    bt[1, 1] = inputs["num_blocks"] + 7
    bad["block_table"] = bt
    res = run_gpu_step(mla, bad, stages=("absorb", "decode", "out"))
    assert res["status"] == mla.MLA_ERR_DEVICE_BOUNDS
    assert np.all(np.isneginf(res["lse"][1]))
    assert np.all(res["o_lat"][1] == 0)
    # sequence 0 is computed normally (no append in either run for this check)
    ref = run_gpu_step(mla, inputs, stages=("absorb", "decode", "out"))
    assert np.array_equal(res["o_lat"][0], ref["o_lat"][0])
    assert good["status"] == 0


def test_seqlen_above_max_reported(mla):
    inputs = synth.random_small(seed=13, H=16, seqlens=[100, 90], Hq=1, **DS)
    res = run_gpu_step(mla, inputs, max_seqlen=95, stages=("absorb", "decode", "out"))
    assert res["status"] == mla.MLA_ERR_DEVICE_BOUNDS
    assert np.all(np.isneginf(res["lse"][0]))
    assert np.all(np.isfinite(res["lse"][1]))
    # the error word is cleared by the read
    ws = mla.alloc_workspace(2, 1, 95, dims_for(mla, inputs))
    assert mla.mla_get_error(ws) == 0


def test_many_items_fall_through_to_cuda_cores(mla):
    """More (sequence, slot) items than the tensor-core plan takes (8192) run
    on the CUDA-core kernel with the same results; sampled sequences are
    compared with the oracle."""
    g = np.random.default_rng(41)
    seqlens = g.integers(1, 70, size=8200).tolist()
    inputs = synth.random_small(seed=41, H=8, seqlens=seqlens, Hq=1, **DS)
    res = run_gpu_step(mla, inputs)
    assert res["status"] == 0
    sample = [0, 1, 4095, 8191, 8192, 8199]
    out, o_lat, lse, _ = run_oracle_step(inputs, sample)
    compare(res["o_lat"][sample], o_lat, "o_lat")
    compare(res["lse"][sample], lse, "lse")
    compare(res["out"][sample], out, "out")
