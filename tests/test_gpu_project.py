"""Parity of the fused projection-and-append step (``mla_project_append``)
against the fp64 oracle: every written cache row equals
``[W_DKV h ; RoPE(W_KR h, p)]`` within the bf16 tolerance, and every other
row of the cache is left bit-identical.
"""

import numpy as np
import pytest
import torch

import synth
from oracle import upstream
from harness import compare

pytestmark = pytest.mark.gpu

D_C, D_R, BS = 512, 64, 64


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mla_latent_kv_74_b300 as m
    return m


def _run(mla, inp, n_new, rope_base=10000.0):
    dev = torch.device("cuda")
    dims = mla.Dims(H=128, d_h=128, d_c=D_C, d_r=D_R, block_size=BS, dtype=torch.bfloat16)
    d = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in inp.items()}
    B, _, d_model = inp["h"].shape
    n = mla.mla_project_append_workspace_size(B, n_new, d_model, dims)
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    cache = d["cache"].clone()
    mla.mla_project_append(d["h"], d["W_DKV"], d["W_KR"], cache, inp["num_blocks"],
                           d["block_table"], d["seqlens"], dims, ws, rope_base=rope_base)
    torch.cuda.synchronize()
    return cache.cpu()


def _check(inp, out, n_new, rope_base=10000.0, what=""):
    """Oracle rows at the written positions; every other row unchanged."""
    theta = upstream.rope_frequencies(D_R, rope_base)
    h = inp["h"].double().numpy()
    W_DKV = inp["W_DKV"].double().numpy()
    W_KR = inp["W_KR"].double().numpy()
    table = inp["block_table"].numpy()
    before = inp["cache"].clone()
    written = np.zeros(before.shape[:2], dtype=bool)
    got, ref = [], []
    for b, s in enumerate(inp["seqlens"].numpy()):
        for i in range(n_new):
            p = int(s) - n_new + i
            if p < 0 or p // BS >= table.shape[1]:
                continue
            blk = int(table[b, p // BS])
            if blk < 0 or blk >= inp["num_blocks"]:
                continue
            written[blk, p % BS] = True
            got.append(out[blk, p % BS].double().numpy())
            ref.append(upstream.cache_row(h[b, i], W_DKV, W_KR, p, theta))
    if got:
        compare(np.stack(got), np.stack(ref), f"project_append rows {what}")
    untouched = torch.from_numpy(~written)
    assert torch.equal(out[untouched], before[untouched]), f"{what}: other rows changed"
    return len(got)


@pytest.mark.parametrize("d_model", [5120, 2048])
def test_project_append_deepseek_dims(mla, d_model):
    seqlens = [1, 64, 65, 700, 4000]
    inp = synth.project_inputs(seed=31, seqlens=seqlens, n_new=1, d_model=d_model)
    out = _run(mla, inp, 1)
    assert _check(inp, out, 1, what=f"d_model={d_model}") == len(seqlens)


def test_project_append_two_new_tokens_and_skips(mla):
    """n_new = 2 (a draft token after the current one); a sequence of length 1
    has its first new position at -1 (skipped); a block entry outside the
    cache is skipped."""
    seqlens = [1, 130, 64, 321]
    inp = synth.project_inputs(seed=32, seqlens=seqlens, n_new=2, d_model=1024)
    inp["block_table"][3, 320 // BS] = inp["num_blocks"] + 5  # position 320: outside
    out = _run(mla, inp, 2)
    # 1 (seq 0) + 2 + 2 + 1 (seq 3 keeps position 319 only)
    assert _check(inp, out, 2, what="n_new=2") == 6


def test_project_append_many_tokens_and_long_positions(mla):
    """300 new tokens (two N tiles of the GEMM) at positions up to 131071,
    where the RoPE angle reaches 1.3e5 rad, and a non-default base."""
    seqlens = [131072] + [512] * 2
    inp = synth.project_inputs(seed=33, seqlens=seqlens, n_new=100, d_model=512)
    out = _run(mla, inp, 100, rope_base=50000.0)
    assert _check(inp, out, 100, rope_base=50000.0, what="long") == 300
