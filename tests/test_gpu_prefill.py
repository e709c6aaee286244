"""Parity of ``mla_prefill`` (standard-order causal prefill: K and V rebuilt
from the latents, then attention over d_h + d_r and d_h) against the fp64
oracle ``oracle.prefill``, whose rows are pinned to the decode oracle.

Tolerance.  Besides the decode path's roundings (P to bf16, the output to
bf16) the standard order rounds the rebuilt K and V to bf16 once, since the
tensor cores take bf16 operands.  An output of magnitude in [4, 8) can thus
carry two half-ulp errors of 2^-6 each, so the max-abs bound here is
2 * 2^-6 = 3.125e-2; the mean-relative bound is the decode path's 5e-3.
"""

import math

import numpy as np
import pytest
import torch

import synth
from oracle import prefill as opf

pytestmark = pytest.mark.gpu

# the decode step's tolerances (bf16 inputs, fp32 accumulation)
MAX_ABS = 2e-2
MEAN_REL = 5e-3
LSE_ABS = 1e-2  # lse is fp32; the scores carry the rounding of K


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mla_latent_kv_74_b300 as m
    return m


def _dims(mla, H):
    return mla.Dims(H=H, d_h=128, d_c=512, d_r=64, block_size=64, dtype=torch.bfloat16)


def _run(mla, t, H, max_seqlen=None, cu_override=None):
    dev = torch.device("cuda")
    g = {k: v.to(dev) for k, v in t.items()}
    if cu_override is not None:
        g["cu_seqlens"] = torch.tensor(cu_override, dtype=torch.int32, device=dev)
    T = g["q_nope"].shape[0]
    cu = g["cu_seqlens"].cpu().numpy()
    if max_seqlen is None:
        max_seqlen = int(np.diff(cu).max()) if len(cu) > 1 else 0
    dims = _dims(mla, H)
    out = torch.full((T, H, 128), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((T, H), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.zeros(mla.mla_prefill_workspace_size(T, dims), dtype=torch.uint8, device=dev)
    mla.mla_prefill(g["q_nope"], g["q_rope"], g["c_kv"], g["k_r"], g["W_UK"], g["W_UV"],
                    g["cu_seqlens"], max_seqlen, dims, out, lse, ws)
    status = mla.mla_get_error(ws)
    return out.float().cpu().numpy(), lse.cpu().numpy(), status


def _np(t):
    return {k: v.double().numpy() if v.dtype != torch.int32 else v.numpy() for k, v in t.items()}


def _check(got, ref, what):
    d = np.abs(got - ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values (rows not written?)"
    max_abs = float(d.max())
    mean_rel = float(d.sum() / np.abs(ref).sum())
    print(f"{what}: max-abs {max_abs:.4g} mean-rel {mean_rel:.4g}")
    assert max_abs <= MAX_ABS, f"{what}: max-abs {max_abs:.3g} > {MAX_ABS}"
    assert mean_rel <= MEAN_REL, f"{what}: mean-rel {mean_rel:.3g} > {MEAN_REL}"


SCALE = 1.0 / math.sqrt(128 + 64)


@pytest.mark.parametrize("seqlens,H", [
    ([1], 4),                    # one token: the output is its own value
    ([77], 4),                   # one ragged key tile
    ([300], 16),                 # three tiles, ragged tail
    ([5, 128, 129, 200], 8),     # packed; a sequence ending exactly on a tile
    ([3, 0, 250], 2),            # an empty sequence in the middle
    ([130, 7], 12),              # a partial last group of heads in the rebuild
    ([1000], 128),               # all DeepSeek-V2 heads, eight tiles
])
def test_prefill_matches_oracle(mla, seqlens, H):
    t = synth.prefill_tensors(seed=7 + H, seqlens=seqlens, H=H)
    got, glse, status = _run(mla, t, H)
    assert status == mla.MLA_OK
    x = _np(t)
    ref, rlse = opf.prefill(x["q_nope"], x["q_rope"], x["c_kv"], x["k_r"], x["W_UK"],
                            x["W_UV"], x["cu_seqlens"], SCALE)
    _check(got, ref, f"out seqlens={seqlens} H={H}")
    assert np.abs(glse - rlse).max() <= LSE_ABS


def test_prefill_max_seqlen_above_lengths(mla):
    # a work list sized for longer prompts: its query tiles past every
    # prompt's end are skipped
    t = synth.prefill_tensors(seed=3, seqlens=[130, 60], H=4)
    got, glse, status = _run(mla, t, 4, max_seqlen=1000)
    assert status == mla.MLA_OK
    x = _np(t)
    ref, rlse = opf.prefill(x["q_nope"], x["q_rope"], x["c_kv"], x["k_r"], x["W_UK"],
                            x["W_UV"], x["cu_seqlens"], SCALE)
    _check(got, ref, "out max_seqlen=1000")


def test_prefill_bad_sequence_is_reported(mla):
    # the second sequence claims 200 tokens against max_seqlen 150: it is
    # skipped and MLA_ERR_DEVICE_BOUNDS recorded; the first is still right
    t = synth.prefill_tensors(seed=5, seqlens=[100, 200], H=2)
    got, glse, status = _run(mla, t, 2, max_seqlen=150)
    assert status == mla.MLA_ERR_DEVICE_BOUNDS
    x = _np(t)
    ref, _ = opf.prefill(x["q_nope"][:100], x["q_rope"][:100], x["c_kv"][:100], x["k_r"][:100],
                         x["W_UK"], x["W_UV"], [0, 100], SCALE)
    _check(got[:100], ref, "out of the valid sequence")
    assert np.isnan(got[100:]).all()  # not written


def test_prefill_full_size_sampled_rows(mla):
    # two 4096-token prompts at H = 128, in the launch configuration the
    # benchmark times; sampled (token, head) rows against the oracle
    seqlens = [4096, 4096]
    H = 128
    t = synth.prefill_tensors(seed=11, seqlens=seqlens, H=H)
    got, glse, status = _run(mla, t, H)
    assert status == mla.MLA_OK
    assert np.all(np.isfinite(got)) and np.all(np.isfinite(glse))
    x = _np(t)
    rng = np.random.default_rng(0)
    heads = [0, 77, 127]
    toks = sorted({0, 1, 127, 128, 129, 2047, 4095} | set(rng.integers(0, 4096, 6).tolist()))
    refs, gots = [], []
    for b, t0 in enumerate((0, 4096)):
        for h in heads:
            for tq in toks:
                o, l = opf.prefill_row(x["q_nope"][t0 + tq, h], x["q_rope"][t0 + tq, h],
                                       x["c_kv"][t0:t0 + tq + 1], x["k_r"][t0:t0 + tq + 1],
                                       x["W_UK"][h], x["W_UV"][h], SCALE)
                refs.append(o)
                gots.append(got[t0 + tq, h])
                assert abs(glse[t0 + tq, h] - l) <= LSE_ABS
    _check(np.stack(gots), np.stack(refs), "sampled rows, 2 x 4096 tokens, H=128")
