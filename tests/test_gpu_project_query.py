"""Parity of the query projections (``mla_project_query``) against the fp64
oracle's ``query_projection``, which the worked example's printed query and
rotated RoPE queries pin."""

import numpy as np
import pytest
import torch

import synth
from harness import compare
from oracle import upstream

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mla_latent_kv_74_b300 as m
    return m


@pytest.mark.parametrize("seqlens,Hq,H,d_model,base", [
    ([8192] * 64, 1, 128, 5120, 10000.0),   # DeepSeek-V2 shape, 64 decode rows
    ([1, 2, 300, 131072], 2, 16, 2048, 10000.0),  # Lite heads, MTP slots, long and empty rows
    ([77, 5], 1, 4, 512, 500.0),            # few heads, another base
])
def test_project_query(mla, seqlens, Hq, H, d_model, base):
    d_h, d_r = 128, 64
    B = len(seqlens)
    t = synth.query_tensors(seed=51 + H, B=B, Hq=Hq, H=H, d_h=d_h, d_r=d_r, d_model=d_model)
    dev = torch.device("cuda")
    dims = mla.Dims(H=H, d_h=d_h, d_c=512, d_r=d_r, block_size=64, dtype=torch.bfloat16)
    sl = torch.tensor(seqlens, dtype=torch.int32)
    q_nope = torch.full((B, Hq, H, d_h), float("nan"), dtype=torch.bfloat16, device=dev)
    q_rope = torch.full((B, Hq, H, d_r), float("nan"), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(mla.mla_project_query_workspace_size(B, Hq, d_model, dims),
                     dtype=torch.uint8, device=dev)
    mla.mla_project_query(t["h"].to(dev), t["W_Q"].to(dev), t["W_QR"].to(dev), sl.to(dev), dims,
                          q_nope, q_rope, ws, rope_base=base)
    torch.cuda.synchronize()
    theta = upstream.rope_frequencies(d_r, base)
    h = t["h"].double().numpy()
    W_Q, W_QR = t["W_Q"].double().numpy(), t["W_QR"].double().numpy()
    ref_n = np.empty((B, Hq, H, d_h))
    ref_r = np.empty((B, Hq, H, d_r))
    for b in range(B):
        for i in range(Hq):
            ref_n[b, i], ref_r[b, i] = upstream.query_projection(
                h[b, i], W_Q, W_QR, H, d_h, d_r, seqlens[b] - Hq + i, theta)
    compare(q_nope.float().cpu().numpy(), ref_n, "q_nope")
    compare(q_rope.float().cpu().numpy(), ref_r, "q_rope")
