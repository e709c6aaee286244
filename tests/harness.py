"""Shared helpers for the GPU parity tests.

``run_gpu_step`` runs one decode step through the C ABI (append, absorb,
decode, out-proj) on the given inputs; ``run_oracle_step`` runs the fp64
oracle on the same inputs for selected sequences.  The two share nothing but
the input tensors from ``synth``.
"""

from __future__ import annotations

import math

import numpy as np
import torch

from oracle import mla as omla

# tolerances stated for the method: bf16 inputs with fp32 accumulation are
# held to max-abs 2e-2 and mean-relative 5e-3; the fp32 tiny workload to 1e-4.
BF16_MAX_ABS = 2e-2
BF16_MEAN_REL = 5e-3
FP32_MAX_ABS = 1e-4


def compare(got, ref, what, dtype="bf16"):
    """max-abs and mean-relative (sum|g-r| / sum|r|) error; -inf must match."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    ninf_r = np.isneginf(ref)
    ninf_g = np.isneginf(got)
    assert np.array_equal(ninf_r, ninf_g), f"{what}: -inf pattern differs"
    fin = ~ninf_r
    assert np.all(np.isfinite(got[fin])), f"{what}: non-finite values"
    if not fin.any():
        return 0.0, 0.0
    d = np.abs(got[fin] - ref[fin])
    max_abs = float(d.max())
    denom = float(np.abs(ref[fin]).sum())
    mean_rel = float(d.sum() / denom) if denom > 0 else 0.0
    if dtype == "bf16":
        assert max_abs <= BF16_MAX_ABS, f"{what}: max-abs {max_abs:.3g} > {BF16_MAX_ABS}"
        assert mean_rel <= BF16_MEAN_REL, f"{what}: mean-rel {mean_rel:.3g} > {BF16_MEAN_REL}"
    else:
        assert max_abs <= FP32_MAX_ABS, f"{what}: max-abs {max_abs:.3g} > {FP32_MAX_ABS}"
    return max_abs, mean_rel


def dims_for(mla, inputs, H=None, d_h=None, d_c=None, d_r=None, block_size=None):
    W = inputs["W_UK"]
    H = H or W.shape[0]
    d_h = d_h or W.shape[1]
    d_c = d_c or W.shape[2]
    d_r = inputs["q_rope"].shape[3] if d_r is None else d_r
    bs = block_size or inputs["cache"].shape[1]
    return mla.Dims(H=H, d_h=d_h, d_c=d_c, d_r=d_r, block_size=bs, dtype=W.dtype)


def to_device(inputs, device="cuda"):
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inputs.items()}


def run_gpu_step(mla, inputs, max_seqlen=None, stages=("append", "absorb", "decode", "out"),
                 ws=None):
    """One step through the binding; returns host copies of every output."""
    dev = to_device(inputs)
    d = dims_for(mla, inputs)
    B, Hq, H, _ = dev["q_nope"].shape
    dt = d.torch_dtype
    if max_seqlen is None:
        max_seqlen = int(inputs["seqlens"].max()) if B else 0
    res = {}
    cache = dev["cache"].clone()
    if "append" in stages:
        mla.mla_append_cache(cache, inputs["num_blocks"], dev["block_table"], dev["seqlens"],
                             dev["c_kv_new"], dev["k_r_new"] if d.d_r else None, d)
    q_lat = torch.empty(B, Hq, H, d.d_c, dtype=dt, device="cuda")
    mla.mla_absorb_query(dev["q_nope"], dev["W_UK"], q_lat, d)
    o_lat = torch.empty(B, Hq, H, d.d_c, dtype=dt, device="cuda")
    lse = torch.empty(B, Hq, H, dtype=torch.float32, device="cuda")
    if ws is None:
        ws = mla.alloc_workspace(B, Hq, max_seqlen, d)
    mla.mla_decode(q_lat, dev["q_rope"] if d.d_r else None, cache, inputs["num_blocks"],
                   dev["block_table"], dev["seqlens"], max_seqlen, d, o_lat, lse, ws)
    out = torch.empty(B, Hq, H, d.d_h, dtype=dt, device="cuda")
    mla.mla_out_proj(o_lat, dev["W_UV"], out, d)
    torch.cuda.synchronize()
    res["status"] = mla.mla_get_error(ws)
    res["cache"] = cache.cpu()
    res["q_lat"] = q_lat.float().cpu().numpy()
    res["o_lat"] = o_lat.float().cpu().numpy()
    res["lse"] = lse.cpu().numpy()
    res["out"] = out.float().cpu().numpy()
    return res


def f64(t):
    return t.double().numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float64)


def compact_sequence(inputs, b):
    """The blocks of sequence ``b`` only, with its table remapped to 0..n-1
    (a plain gather, so the oracle need not hold the whole cache in fp64)."""
    bs = inputs["cache"].shape[1]
    n = int(inputs["seqlens"][b])
    nblk = max(1, -(-n // bs))
    phys = inputs["block_table"][b, :nblk].long()
    cache = f64(inputs["cache"][phys])
    return cache, np.arange(nblk)[None, :]


def run_oracle_step(inputs, batch_indices=None, scale=None, head_indices=None):
    """fp64 oracle on the same inputs: append, then the un-absorbed decode.

    Returns ``out, o_lat, lse`` for ``batch_indices`` and the oracle's
    ``q_lat`` for all rows.
    """
    B, Hq = inputs["q_nope"].shape[:2]
    if batch_indices is None:
        batch_indices = list(range(B))
    d_c = inputs["W_UK"].shape[2]
    W_UK = f64(inputs["W_UK"])
    W_UV = f64(inputs["W_UV"])
    outs, olats, lses = [], [], []
    for b in batch_indices:
        cache, table = compact_sequence(inputs, b)
        sl = inputs["seqlens"][b:b + 1].numpy()
        cache = omla.append_to_cache(cache, table, sl, f64(inputs["c_kv_new"][b:b + 1]),
                                     f64(inputs["k_r_new"][b:b + 1]))
        o, ol, ls = omla.mla_decode(f64(inputs["q_nope"][b:b + 1]),
                                    f64(inputs["q_rope"][b:b + 1]), cache, table, sl, W_UK, W_UV,
                                    Hq, scale=scale, head_indices=head_indices)
        outs.append(o)
        olats.append(ol)
        lses.append(ls)
    q_lat = omla.absorb_query(f64(inputs["q_nope"]), W_UK)
    return (np.concatenate(outs), np.concatenate(olats), np.concatenate(lses), q_lat)


def tiny_inputs():
    """The tiny fp32 workload: hidden states and weights from ``synth``,
    turned into cache rows and queries by the oracle's upstream projections,
    rounded once to fp32 (the values both sides then consume)."""
    import synth
    from oracle import upstream

    raw = synth.make_tiny_raw()
    w = raw["workload"]
    rows, q_nope, q_rope = upstream.tiny_workload_inputs(raw["h"], raw["W_DKV"], raw["W_KR"],
                                                         raw["W_Q"], raw["W_QR"], w.H, w.d_h,
                                                         w.d_r)
    T = w.seqlen
    f = lambda x: torch.tensor(np.asarray(x), dtype=torch.float32)
    cache = torch.zeros(1, 64, w.D, dtype=torch.float32)
    cache[0, :T - 1] = f(rows[:T - 1])  # the newest token is appended by the step
    return {
        "cache": cache,
        "c_kv_new": f(rows[T - 1:, :w.d_c])[None],
        "k_r_new": f(rows[T - 1:, w.d_c:])[None],
        "q_nope": f(q_nope)[None, None],
        "q_rope": f(q_rope)[None, None],
        "W_UK": f(raw["W_UK"]),
        "W_UV": f(raw["W_UV"]),
        "block_table": torch.zeros(1, 1, dtype=torch.int32),
        "seqlens": torch.tensor([T], dtype=torch.int32),
        "num_blocks": 1,
    }
