"""Parity of the output projection over the concatenated heads
(``mla_o_proj``) against the fp64 oracle's ``output_projection``, which the
worked example's printed ``u_4`` pins."""

import numpy as np
import pytest
import torch

import synth
from harness import compare
from oracle import mla as omla

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mla_latent_kv_74_b300 as m
    return m


def _run(mla, t, H, d_h):
    dev = torch.device("cuda")
    B, Hq = t["out"].shape[:2]
    d_model = t["W_O"].shape[0]
    dims = mla.Dims(H=H, d_h=d_h, d_c=512, d_r=64, block_size=64, dtype=torch.bfloat16)
    out, W_O = t["out"].to(dev), t["W_O"].to(dev)
    u = torch.full((B, Hq, d_model), float("nan"), dtype=torch.bfloat16, device=dev)
    n = mla.mla_o_proj_workspace_size(B, Hq, d_model, dims)
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    mla.mla_o_proj(out, W_O, u, dims, ws)
    torch.cuda.synchronize()
    return u.float().cpu().numpy()


def _oracle(t):
    out = t["out"].double().numpy()
    B, Hq = out.shape[:2]
    W_O_rows = t["W_O"].double().numpy().T  # the oracle's row-vector form [H*d_h, d]
    return np.stack([np.stack([omla.output_projection(out[b, i], W_O_rows)
                               for i in range(Hq)]) for b in range(B)])


@pytest.mark.parametrize("B,Hq,H,d_model", [
    (64, 1, 128, 5120),   # DeepSeek-V2: 64 decode rows, 16384 -> 5120
    (3, 1, 128, 5120),    # a 16-row N tile, mostly empty
    (150, 2, 16, 2048),   # V2-Lite heads, 300 rows: two N tiles
    (5, 1, 8, 1000),      # d_model not a multiple of the 128-row M tile
])
def test_o_proj(mla, B, Hq, H, d_model):
    t = synth.o_proj_tensors(seed=41 + H, B=B, Hq=Hq, H=H, d_h=128, d_model=d_model)
    got = _run(mla, t, H, 128)
    compare(got, _oracle(t), f"u B={B} Hq={Hq} H={H} d_model={d_model}")
