"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times (same entry points, same max_seqlen = max(seqlens)).

The oracle cannot redo a whole workload in seconds, so each test checks every
output for properties that hold at any size (finite, right -inf pattern,
q_lat everywhere) and compares sampled (sequence, head) rows one by one
against the fp64 oracle.
"""

import numpy as np
import pytest
import torch

import synth
from harness import compare, run_gpu_step, run_oracle_step

pytestmark = pytest.mark.gpu

# workload -> (sampled sequences, sampled heads or None for all)
SAMPLES = {
    "lite": ([0, 31], None),
    "v2": ([0, 63], list(range(0, 128, 4))),
    "mtp": (None, list(range(0, 128, 8))),  # the longest and the shortest sequence
    "long": ([2], list(range(0, 128, 16))),
}


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mla_latent_kv_74_b300 as m
    return m


@pytest.mark.parametrize("name", ["lite", "v2", "mtp", "long"])
def test_full_size_sampled(mla, name):
    inputs = synth.make_bf16_inputs(name)
    res = run_gpu_step(mla, inputs)
    assert res["status"] == 0
    assert np.all(np.isfinite(res["lse"])), "every row sees at least one token"
    assert np.all(np.isfinite(res["o_lat"])) and np.all(np.isfinite(res["out"]))
    seqs, heads = SAMPLES[name]
    if seqs is None:
        sl = inputs["seqlens"].numpy()
        seqs = [int(np.argmax(sl)), int(np.argmin(sl))]
    out, o_lat, lse, q_lat = run_oracle_step(inputs, seqs, head_indices=heads)
    hs = list(range(inputs["W_UK"].shape[0])) if heads is None else heads
    compare(res["q_lat"], q_lat, f"{name} q_lat (all rows)")
    g = lambda k: res[k][seqs][:, :, hs]
    compare(g("o_lat"), o_lat, f"{name} o_lat")
    compare(g("lse"), lse, f"{name} lse")
    compare(g("out"), out, f"{name} out")
