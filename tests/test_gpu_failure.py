"""The failure path on the GPU without a fault: a bounded wait that nothing
satisfies gives up, the kernel records MLA_ERR_TIMEOUT in the workspace's
error word, ``mla_get_error`` reports and clears it, and the same context
then runs a decode that matches the oracle."""

import pytest
import torch

import synth
from harness import compare, run_gpu_step, run_oracle_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mla_latent_kv_74_b300 as m
    return m


def test_lost_wait_is_reported_and_the_context_stays_usable(mla):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    mla.mla_selftest_lost_wait(ws)
    assert mla.mla_get_error(ws) == mla.MLA_ERR_TIMEOUT
    assert mla.mla_get_error(ws) == mla.MLA_OK  # read once, then cleared
    inp = synth.random_small(seed=4, H=16, d_h=128, d_c=512, d_r=64, seqlens=[70, 3], Hq=1)
    res = run_gpu_step(mla, inp)
    assert res["status"] == mla.MLA_OK
    out, o_lat, lse, q_lat = run_oracle_step(inp)
    compare(res["o_lat"], o_lat, "o_lat after the lost wait", "bf16")
    compare(res["out"], out, "out after the lost wait", "bf16")
