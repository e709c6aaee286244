"""mla_decode_noalloc, the decode entry point for callers that cannot allocate.

Some callers cannot call cudaMalloc (a plugin whose host application owns the
device memory, a serving loop that must not block on an allocation), so they
cannot hand mla_decode a workspace.  mla_decode_noalloc takes the workspace
from a fixed array inside the library instead.  These tests call it through
the C ABI and check that two calls in a row give the same results as
mla_decode with a caller-provided workspace, within the tolerances every
parity test here uses.  The file is named to run last, so a failure here
cannot hide the rest of the suite.
"""

import ctypes


import numpy as np
import pytest
import torch

import synth
from harness import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mla_latent_kv_74_b300 as m
    return m


def _run_both(mla, inputs, dtype):
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inputs.items()}
    B, Hq, H, d_h = dev["q_nope"].shape
    d_c = dev["W_UK"].shape[2]
    d_r = dev["q_rope"].shape[3]
    dims = mla.Dims(H=H, d_h=d_h, d_c=d_c, d_r=d_r, block_size=dev["cache"].shape[1],
                    dtype=dev["W_UK"].dtype)
    max_seqlen = int(inputs["seqlens"].max())
    q_lat = torch.empty(B, Hq, H, d_c, dtype=dev["W_UK"].dtype, device="cuda")
    mla.mla_absorb_query(dev["q_nope"], dev["W_UK"], q_lat, dims)
    # the existing entry point, with a workspace the caller allocates
    ws = mla.alloc_workspace(B, Hq, max_seqlen, dims)
    o_ref = torch.empty_like(q_lat)
    lse_ref = torch.empty(B, Hq, H, dtype=torch.float32, device="cuda")
    mla.mla_decode(q_lat, dev["q_rope"], dev["cache"], inputs["num_blocks"], dev["block_table"],
                   dev["seqlens"], max_seqlen, dims, o_ref, lse_ref, ws)
    torch.cuda.synchronize()
    lib = mla.raw_lib()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):  # the scratch keeps the previous call's contents
        o = torch.full_like(q_lat, float("nan"))
        lse = torch.full((B, Hq, H), float("nan"), dtype=torch.float32, device="cuda")
        status = lib.mla_decode_noalloc(
            q_lat.data_ptr(), dev["q_rope"].data_ptr(), dev["cache"].data_ptr(),
            inputs["num_blocks"], dev["block_table"].data_ptr(), dev["block_table"].shape[1],
            dev["seqlens"].data_ptr(), max_seqlen, B, Hq, ctypes.byref(dims), o.data_ptr(),
            lse.data_ptr(), stream)
        assert status == mla.MLA_OK, mla.status_string(status)
        torch.cuda.synchronize()
        compare(o.float().cpu().numpy(), o_ref.float().cpu().numpy(), f"o_lat call {call}", dtype)
        compare(lse.cpu().numpy(), lse_ref.cpu().numpy(), f"lse call {call}", dtype)


def test_noalloc_matches_decode_tensor_core_path(mla):
    inputs = synth.random_small(seed=31, H=128, d_h=128, d_c=512, d_r=64,
                                seqlens=[300, 1000, 64, 1], Hq=1)
    _run_both(mla, inputs, "bf16")


def test_noalloc_matches_decode_causal_slots(mla):
    inputs = synth.random_small(seed=32, H=128, d_h=128, d_c=512, d_r=64,
                                seqlens=[700, 65, 2], Hq=2)
    _run_both(mla, inputs, "bf16")


def test_noalloc_matches_decode_cuda_core_path(mla):
    inputs = synth.random_small(seed=33, H=8, d_h=32, d_c=64, d_r=32, seqlens=[17, 100, 40],
                                Hq=2, block_size=32, dtype=torch.float32)
    _run_both(mla, inputs, "fp32")


def test_noalloc_rejects_oversized_problem(mla):
    """A problem whose workspace would exceed the built-in array is refused
    before anything is launched."""
    dims = mla.Dims(H=64, d_h=128, d_c=512, d_r=64, block_size=64, dtype=torch.float32)
    B, Hq, max_seqlen = 512, 1, 65536
    assert mla.mla_decode_workspace_size(B, Hq, max_seqlen, dims) > mla.NOALLOC_SCRATCH_BYTES
    p = ctypes.c_void_p(1 << 20)
    status = mla.raw_lib().mla_decode_noalloc(p, p, p, 1, p, 1, p, max_seqlen, B, Hq,
                                              ctypes.byref(dims), p, p, None)
    assert status == mla.MLA_ERR_WORKSPACE


def _noalloc(mla, dev, inputs, q_lat, dims, o, lse):
    return mla.raw_lib().mla_decode_noalloc(
        q_lat.data_ptr(), dev["q_rope"].data_ptr(), dev["cache"].data_ptr(), inputs["num_blocks"],
        dev["block_table"].data_ptr(), dev["block_table"].shape[1], dev["seqlens"].data_ptr(),
        int(inputs["seqlens"].max()), q_lat.shape[0], q_lat.shape[1], ctypes.byref(dims),
        o.data_ptr(), lse.data_ptr(), torch.cuda.current_stream().cuda_stream)


def test_noalloc_reports_device_errors_then_recovers(mla):
    """A block-table entry outside [0, num_blocks) is caught on the device:
    mla_decode_noalloc_get_error returns MLA_ERR_DEVICE_BOUNDS (and clears it),
    that sequence's rows come back as o_lat = 0, lse = -inf, the other
    sequence is unaffected, and the next clean call through the same shared
    array matches mla_decode again."""
    inputs = synth.random_small(seed=34, H=128, d_h=128, d_c=512, d_r=64, seqlens=[130, 200],
                                Hq=1)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inputs.items()}
    dims = mla.Dims(H=128, d_h=128, d_c=512, d_r=64, block_size=64, dtype=torch.bfloat16)
    q_lat = torch.empty(2, 1, 128, 512, dtype=torch.bfloat16, device="cuda")
    mla.mla_absorb_query(dev["q_nope"], dev["W_UK"], q_lat, dims)
    ws = mla.alloc_workspace(2, 1, int(inputs["seqlens"].max()), dims)
    o_ref = torch.empty_like(q_lat)
    lse_ref = torch.empty(2, 1, 128, dtype=torch.float32, device="cuda")
    mla.mla_decode(q_lat, dev["q_rope"], dev["cache"], inputs["num_blocks"], dev["block_table"],
                   dev["seqlens"], int(inputs["seqlens"].max()), dims, o_ref, lse_ref, ws)
    assert mla.mla_get_error(ws) == mla.MLA_OK

    bad = dict(dev)
    bt = dev["block_table"].clone()
    bt[1, 1] = inputs["num_blocks"] + 7
    bad["block_table"] = bt
    o = torch.full_like(q_lat, float("nan"))
    lse = torch.full((2, 1, 128), float("nan"), dtype=torch.float32, device="cuda")
    assert _noalloc(mla, bad, inputs, q_lat, dims, o, lse) == mla.MLA_OK
    assert mla.mla_decode_noalloc_get_error() == mla.MLA_ERR_DEVICE_BOUNDS
    assert mla.mla_decode_noalloc_get_error() == mla.MLA_OK  # read and cleared
    o_h, lse_h = o.float().cpu().numpy(), lse.cpu().numpy()
    assert np.all(o_h[1] == 0) and np.all(np.isneginf(lse_h[1]))
    assert np.array_equal(o_h[0], o_ref.float().cpu().numpy()[0])
    assert np.array_equal(lse_h[0], lse_ref.cpu().numpy()[0])

    o2 = torch.full_like(q_lat, float("nan"))
    lse2 = torch.full((2, 1, 128), float("nan"), dtype=torch.float32, device="cuda")
    assert _noalloc(mla, dev, inputs, q_lat, dims, o2, lse2) == mla.MLA_OK
    assert mla.mla_decode_noalloc_get_error() == mla.MLA_OK
    compare(o2.float().cpu().numpy(), o_ref.float().cpu().numpy(), "o_lat after an error", "bf16")
    compare(lse2.cpu().numpy(), lse_ref.cpu().numpy(), "lse after an error", "bf16")


def test_noalloc_takes_the_ragged_two_slot_shape(mla):
    """The workspace of the ragged two-slot workload (B = 128, Hq = 2,
    max_seqlen 32768, H = 128) fits the built-in array."""
    dims = mla.Dims(H=128, d_h=128, d_c=512, d_r=64, block_size=64, dtype=torch.bfloat16)
    assert mla.mla_decode_workspace_size(128, 2, 32768, dims) <= mla.NOALLOC_SCRATCH_BYTES
