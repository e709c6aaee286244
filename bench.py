"""Benchmark of one MLA decode step (append + absorb + decode + out-proj).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload v2]
    python bench.py --impl reference ...     # the fp64 CPU oracle, timed

Default workload: the DeepSeek-V2-shaped paged decode (H=128, d_h=128,
d_c=512, d_r=64, B=64, seqlen 8192, Hq=1, block 64, permuted block table),
seeded synthetic data.  Prints ONE JSON line on rank 0.

Timing: W untimed warm-up steps, then K steps.  Before every timed step L2
is flushed by writing a 256 MiB buffer (outside the step's events); each
step is timed with CUDA events on the stream the library launches on.  The
mla_decode call is also timed on its own: that is the kernel the roofline
fraction describes.  N > 1 (under torchrun, or ``--gpus N`` alone, which
starts the N rank processes itself): every rank runs its own replica of the
workload on its own GPU (weak scaling, no collective on the data path); rank
0 reports the max over ranks and the whole-job throughput.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MLA decode TFLOP/s + latent-cache GB/s, fraction of 1×B300 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
L2_FLUSH_BYTES = 256 << 20


# ---------------------------------------------------------------------------
# algorithmic work (the method's own counts, not the kernels')
# ---------------------------------------------------------------------------


def visible_tokens(seqlens, Hq):
    """sum over sequences and query slots of the visible cache length."""
    s = np.asarray(seqlens, np.int64)
    return int(sum(np.maximum(0, s - Hq + i + 1).sum() for i in range(Hq)))


def max_over_ranks(values, world, device=None):
    """The element-wise maximum of ``values`` over all ranks (the slowest
    replica sets the whole job's time).  NCCL reduces device tensors, gloo
    host tensors."""
    if world <= 1:
        return [float(v) for v in values]
    on_dev = device is not None and torch.distributed.get_backend() == "nccl"
    t = torch.tensor([float(v) for v in values], dtype=torch.float64,
                     device=device if on_dev else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.cpu().tolist()


def whole_job_rate(work_per_rank, world, ms):
    """Throughput of ``world`` replicas that each did ``work_per_rank`` units,
    the slowest in ``ms`` milliseconds (weak scaling): units per second."""
    return world * work_per_rank / (ms * 1e-3)


def decode_work(w, seqlens):
    """FLOPs and bytes of mla_decode: QK^T over d_c + d_r and P C over d_c
    per visible (token, query slot) and head; bytes are the cache rows read
    once per sequence plus q_lat/q_rope in and o_lat/lse out."""
    vt = visible_tokens(seqlens, w.Hq)
    flops = 2 * w.H * (w.d_c + w.d_r) * vt + 2 * w.H * w.d_c * vt
    cache_tokens = int(np.asarray(seqlens, np.int64).sum())
    rows = len(seqlens) * w.Hq * w.H
    bytes_ = cache_tokens * (w.d_c + w.d_r) * 2 + rows * (w.d_c + w.d_r) * 2 + rows * (w.d_c * 2 + 4)
    return flops, bytes_


def gemm_work(w, B):
    rows = B * w.Hq
    flops = 2 * rows * w.H * w.d_h * w.d_c
    bytes_ = w.H * w.d_h * w.d_c * 2 + rows * w.H * (w.d_h + w.d_c) * 2
    return flops, bytes_


def prefill_work(seqlens, H, d_h=128, d_r=64, d_c=512):
    """Tensor FLOPs of mla_prefill: rebuilding [K_nope | V] (``2·T·H·2d_h·d_c``)
    and the causal attention (``2·H·(d_h + d_r + d_h)`` per visible
    (query, key) pair, ``T_b (T_b + 1) / 2`` pairs per prompt)."""
    T = int(sum(seqlens))
    kv = 2 * T * H * 2 * d_h * d_c
    attn = sum(int(n) * (int(n) + 1) // 2 for n in seqlens) * 2 * H * (2 * d_h + d_r)
    return kv, attn


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.25)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------


def setup_inputs(name, device, batch=None):
    inp = synth.make_bf16_inputs(name, B_override=batch)
    dev = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    return inp, dev


def run_ours(args, rank, world, device):
    import mla_latent_kv_74_b300 as mla

    w = synth.WORKLOADS[args.workload]
    inp, dev = setup_inputs(args.workload, device, args.batch)
    w = inp["workload"]
    B = w.B
    seqlens = inp["seqlens"].numpy()
    max_seqlen = int(seqlens.max())
    dims = mla.Dims(H=w.H, d_h=w.d_h, d_c=w.d_c, d_r=w.d_r, block_size=w.block_size,
                    dtype=torch.bfloat16)
    cache = dev["cache"]
    q_lat = torch.empty(B, w.Hq, w.H, w.d_c, dtype=torch.bfloat16, device=device)
    o_lat = torch.empty_like(q_lat)
    lse = torch.empty(B, w.Hq, w.H, dtype=torch.float32, device=device)
    out = torch.empty(B, w.Hq, w.H, w.d_h, dtype=torch.bfloat16, device=device)
    ws = mla.alloc_workspace(B, w.Hq, max_seqlen, dims, device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def step(x, o=None):
        # nothing between the calls: consecutive kernels of the step overlap
        # (programmatic dependent launch), which an event record would stop
        mla.mla_append_cache(cache, inp["num_blocks"], x["block_table"], x["seqlens"],
                             x["c_kv_new"], x["k_r_new"], dims, stream)
        mla.mla_absorb_query(x["q_nope"], dev["W_UK"], q_lat, dims, stream)
        mla.mla_decode(q_lat, x["q_rope"], cache, inp["num_blocks"], x["block_table"],
                       x["seqlens"], max_seqlen, dims, o_lat, lse, ws, stream)
        mla.mla_out_proj(o_lat, dev["W_UV"], out if o is None else o, dims, stream)

    # ---- device-resident timing -------------------------------------------
    # All timed steps are enqueued before one synchronisation, so the GPU
    # never idles between a step's kernels waiting for the host to prepare
    # the next call (that gap would land inside the measured intervals).
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for _ in range(args.warmup):
        flush.zero_()
        step(dev)
    torch.cuda.synchronize()
    status = mla.mla_get_error(ws)
    if status != 0:
        raise RuntimeError(f"device error after warm-up: {mla.status_string(status)}")

    step_ms, dec_ms = [], []
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(smi_index(device.index)) as clocks:
        t_wall = time.perf_counter()
        # A spin kernel ahead of the timed steps (outside every event pair)
        # gives the host time to enqueue them all, so no measured interval
        # contains the GPU waiting for the next launch (about 1 ms per step).
        torch.cuda._sleep(int(min(2e9, 2e6 * args.steps)))
        for it in range(args.steps):
            ev = evs[it]
            flush.zero_()
            ev[0].record(stream)
            step(dev)
            ev[1].record(stream)
        torch.cuda.synchronize()
        for ev in evs:
            step_ms.append(ev[0].elapsed_time(ev[1]))
        t_wall = time.perf_counter() - t_wall
        # mla_decode alone (the call the roofline describes), same inputs,
        # L2 flushed before every call
        dec_ms.append(_time_calls(
            lambda: mla.mla_decode(q_lat, dev["q_rope"], cache, inp["num_blocks"],
                                   dev["block_table"], dev["seqlens"], max_seqlen, dims, o_lat,
                                   lse, ws, stream), args.steps, flush, stream))
    if world > 1:
        torch.distributed.barrier()
    status = mla.mla_get_error(ws)
    if status != 0:
        raise RuntimeError(f"device error in the timed region: {mla.status_string(status)}")

    # ---- end to end through host buffers ------------------------------------
    # Every step's inputs sit in a pinned host buffer (each tensor at a
    # 256-byte aligned offset) and go up in one copy; its output comes back
    # in one copy.  Two forms are timed:
    #  * pipelined (the reported value): as a serving loop runs, step k's
    #    upload (one copy stream) and step k-1's download (another) overlap
    #    the compute; inputs and outputs are triple-buffered (a 3.25 MB
    #    upload from a buffer the CPU has written can take as long as a
    #    step), and one event pair spans all the steps, every upload and
    #    every download;
    #  * serial: upload, step, download, then the host waits, every step.
    host_keys = ("q_nope", "q_rope", "c_kv_new", "k_r_new", "block_table", "seqlens")
    offs, total = {}, 0
    for k in host_keys:
        offs[k] = total
        total += (inp[k].numel() * inp[k].element_size() + 255) // 256 * 256
    nbuf = 3
    host_bufs = [torch.empty(total, dtype=torch.uint8, pin_memory=True) for _ in range(nbuf)]
    dev_bufs = [torch.empty(total, dtype=torch.uint8, device=device) for _ in range(nbuf)]
    staged = [{} for _ in range(nbuf)]
    for i in range(nbuf):
        for k in host_keys:
            t = inp[k].contiguous()
            n = t.numel() * t.element_size()
            host_bufs[i][offs[k]:offs[k] + n].copy_(t.reshape(-1).view(torch.uint8))
            staged[i][k] = dev_bufs[i][offs[k]:offs[k] + n].view(t.dtype).view(t.shape)
    outs = [out] + [torch.empty_like(out) for _ in range(nbuf - 1)]
    # The inputs were just written by the CPU, so their lines sit dirty in
    # its caches, and a DMA read of such a buffer runs at a fraction of the
    # link rate (180-520 us for 3.25 MB against ~64 us).  Writing a buffer
    # larger than the host's caches once moves them out, as for inputs written
    # well before their step.
    _evict = torch.empty(512 << 20, dtype=torch.uint8)
    _evict.fill_(1)
    del _evict
    out_hosts = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(nbuf)]
    h2d = total
    d2h = out_hosts[0].numel() * out_hosts[0].element_size()
    up, down = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev_up, ev_done, ev_down = ([torch.cuda.Event() for _ in range(nbuf)] for _ in range(3))

    def run_pipelined(n):
        """Mean ms per step of n steps with the copies overlapping the compute."""
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        torch.cuda._sleep(int(min(2e9, 2e6 * n)))  # the host enqueues every step first
        t0.record(stream)
        up.wait_stream(stream)
        down.wait_stream(stream)
        for it in range(n):
            b = it % nbuf
            if it >= nbuf:  # the step that last read this input slot is done
                up.wait_event(ev_done[b])
            with torch.cuda.stream(up):
                dev_bufs[b].copy_(host_bufs[b], non_blocking=True)
            ev_up[b].record(up)
            stream.wait_event(ev_up[b])
            if it >= nbuf:  # this output slot's previous download is done
                stream.wait_event(ev_down[b])
            step(staged[b], outs[b])
            ev_done[b].record(stream)
            down.wait_event(ev_done[b])
            with torch.cuda.stream(down):
                out_hosts[b].copy_(outs[b], non_blocking=True)
            ev_down[b].record(down)
        stream.wait_stream(down)
        t1.record(stream)
        t1.synchronize()
        return t0.elapsed_time(t1) / n

    run_pipelined(args.warmup)
    e2e_pipe_ms = run_pipelined(args.steps)
    e2e_ms = []
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for it in range(args.warmup + args.steps):
        flush.zero_()
        e0.record(stream)
        dev_bufs[0].copy_(host_bufs[0], non_blocking=True)
        step(staged[0])
        out_hosts[0].copy_(out, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        if it >= args.warmup:
            e2e_ms.append(e0.elapsed_time(e1))
    status = mla.mla_get_error(ws)
    if status != 0:
        raise RuntimeError(f"device error in the end-to-end steps: {mla.status_string(status)}")

    # ---- the other decode workloads (mla_decode alone) -------------------------
    configs = measure_other_configs(mla, args, flush, stream, device) if rank == 0 else None

    # ---- the fused projection-and-append step (measured on its own) ---------
    proj = measure_project_append(mla, args, w, dev, inp, dims, flush, stream, device)
    oproj = measure_o_proj(mla, args, w, out, dims, flush, stream, device)
    qproj = measure_project_query(mla, args, w, dev, dims, flush, stream, device)
    pre = measure_prefill(mla, args, w, flush, stream, device)

    # ---- reduce over ranks ----------------------------------------------------
    t_step, t_dec, t_e2e, t_e2e_serial = max_over_ranks(
        [float(np.mean(step_ms)), float(np.mean(dec_ms)), e2e_pipe_ms, float(np.mean(e2e_ms))],
        world, device)
    if rank != 0:
        return None

    dflops, dbytes = decode_work(w, seqlens)
    gflops, gbytes = gemm_work(w, B)
    step_flops = dflops + 2 * gflops
    peaks, peak_src = load_peaks()
    hbm = peaks["hbm_gbs"]
    tc_burst = peaks["bf16_tflops"]
    dec_gbs = dbytes / (t_dec * 1e-3) / 1e9
    dec_tflops = dflops / (t_dec * 1e-3) / 1e12
    t_roof = max(dbytes / (hbm * 1e9), dflops / (tc_burst * 1e12))
    bound = "hbm" if dbytes / (hbm * 1e9) >= dflops / (tc_burst * 1e12) else "tensor"
    achieved, peak, unit = (dec_gbs, hbm, "GB/s") if bound == "hbm" else (dec_tflops, tc_burst,
                                                                         "TFLOP/s")
    value = whole_job_rate(step_flops, world, t_step) / 1e12
    launches_per_step = 1 + 1 + decode_launches(mla, dims, w) + 1
    traffic = load_traffic(args.workload)
    res = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) latents/queries, N(0,1/512) weights; no trained weights)",
        "config": {
            "workload": synth.DESCRIPTIONS[args.workload]
            + ("" if args.batch is None else f" (batch overridden to {B})"),
            "name": args.workload,
            "B": B, "Hq": w.Hq, "H": w.H, "d_h": w.d_h, "d_c": w.d_c, "d_r": w.d_r,
            "block_size": w.block_size,
            "seqlen": int(max_seqlen) if w.seqlen else "ragged",
            "visible_tokens": visible_tokens(seqlens, w.Hq),
            "step": "append + absorb + decode(split-KV + combine) + out_proj",
            "l2": "flushed before every timed step (256 MiB write outside the step's events)",
            "parallelism": (f"dp{world}: one replica of the workload per GPU (weak scaling, "
                            "no collective on the data path)") if world > 1 else "single GPU",
        },
        "decode": {
            "ms": round(t_dec, 5),
            "tflops": round(dec_tflops, 2),
            "cache_gbs": round(dec_gbs, 1),
            "roofline_time_ms": round(t_roof * 1e3, 5),
            "roofline_time_frac": round(t_roof / (t_dec * 1e-3), 4),
            "tensor_frac_of_burst": round(dec_tflops / tc_burst, 4),
            "tensor_frac_of_sustained": round(dec_tflops / peaks["bf16_tflops_sustained"], 4),
            "algorithmic_flops": dflops,
            "algorithmic_bytes": dbytes,
        },
        "roofline": {
            "kernel": "mla_decode",
            "bound": bound,
            "achieved": round(achieved, 2),
            "peak": peak,
            "unit": unit,
            "frac": round(achieved / peak, 4),
            "peak_source": f"{peak_src} ({'burst' if bound == 'tensor' else 'copy'})",
            "traffic": traffic,
        },
        "e2e": {
            "value": round(whole_job_rate(step_flops, world, t_e2e) / 1e12, 3),
            "unit": "TFLOP/s",
            "ms_per_step": round(t_e2e, 5),
            "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h),
            "form": "pipelined: each step's upload and the previous step's download "
                    "overlap the compute (two copy streams, triple-buffered); no L2 flush "
                    "between steps, the 604 MB cache stream is larger than L2",
            "serial_ms_per_step": round(t_e2e_serial, 5),
        },
        "gpu_launches": int(launches_per_step * args.steps),
        "clocks": clocks.summary(),
        "wall_s_timed_region": round(t_wall, 3),
    }
    if configs:
        res["configs"] = configs
    if proj is not None:
        res["project_append"] = proj
    if oproj is not None:
        res["o_proj"] = oproj
    if qproj is not None:
        res["project_query"] = qproj
    if pre is not None:
        res["prefill"] = pre
    return res


# workloads whose mla_decode is measured beside the step's (tiny is a
# parity case: launch-bound, nothing to fraction)
OTHER_CONFIGS = ("lite", "mtp", "long")


def measure_other_configs(mla, args, flush, stream, device, names=OTHER_CONFIGS, batch=None):
    """``mla_decode`` alone on each of the other workloads, with its own
    inputs (the same seeded recipe as the parity tests), L2 flushed before
    every call: time, cache GB/s, TFLOP/s and the fraction of
    ``max(bytes / HBM, FLOPs / bf16 peak)``, the same roofline as the step's."""
    peaks, _ = load_peaks()
    out = {}
    for name in names:
        if name == args.workload:
            continue
        inp, dev = setup_inputs(name, device, batch)
        w = inp["workload"]
        seqlens = inp["seqlens"].numpy()
        max_seqlen = int(seqlens.max())
        dims = mla.Dims(H=w.H, d_h=w.d_h, d_c=w.d_c, d_r=w.d_r, block_size=w.block_size,
                        dtype=torch.bfloat16)
        q_lat = torch.empty(w.B, w.Hq, w.H, w.d_c, dtype=torch.bfloat16, device=device)
        mla.mla_absorb_query(dev["q_nope"], dev["W_UK"], q_lat, dims, stream)
        o_lat = torch.empty_like(q_lat)
        lse = torch.empty(w.B, w.Hq, w.H, dtype=torch.float32, device=device)
        ws = mla.alloc_workspace(w.B, w.Hq, max_seqlen, dims, device=device)

        def call():
            mla.mla_decode(q_lat, dev["q_rope"], dev["cache"], inp["num_blocks"],
                           dev["block_table"], dev["seqlens"], max_seqlen, dims, o_lat, lse, ws,
                           stream)

        ms = _time_calls(call, max(3, min(args.steps, 20)), flush, stream)
        status = mla.mla_get_error(ws)
        if status != 0:
            raise RuntimeError(f"{name}: device error {mla.status_string(status)}")
        flops, nbytes = decode_work(w, seqlens)
        t_mem, t_tc = nbytes / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops"] * 1e12)
        out[name] = {
            "workload": synth.DESCRIPTIONS[name] + ("" if batch is None else f" (batch {w.B})"),
            "ms": round(ms, 5),
            "cache_gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
            "tflops": round(flops / (ms * 1e-3) / 1e12, 2),
            "bound": "hbm" if t_mem >= t_tc else "tensor",
            "roofline_time_ms": round(max(t_mem, t_tc) * 1e3, 5),
            "roofline_time_frac": round(max(t_mem, t_tc) / (ms * 1e-3), 4),
            "algorithmic_flops": flops,
            "algorithmic_bytes": nbytes,
            "traffic": load_traffic(name),
        }
        del inp, dev, q_lat, o_lat, lse, ws
        torch.cuda.empty_cache()
    return out


# hidden size of the model each workload is shaped after (DeepSeek-V2: 5120,
# V2-Lite: 2048), for the fused projection-and-append measurement
PROJ_D_MODEL = {"v2": 5120, "mtp": 5120, "long": 5120, "lite": 2048}


def _time_calls(call, n, flush, stream):
    """Mean CUDA-event time of ``n`` calls, L2 flushed before each, all
    enqueued behind a spin kernel; three untimed calls first."""
    for _ in range(3):
        flush.zero_()
        call()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    torch.cuda.synchronize()
    torch.cuda._sleep(int(2e6 * n))
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        call()
        e1.record(stream)
    torch.cuda.synchronize()
    return float(np.mean([e0.elapsed_time(e1) for e0, e1 in evs]))


def measure_project_query(mla, args, w, dev, dims, flush, stream, device):
    """``mla_project_query`` for the step's B * Hq query rows at the model's
    hidden size.  Algorithmic bytes: ``W_Q`` and ``W_QR`` once, ``h`` in,
    ``q_nope`` and ``q_rope`` out; FLOPs ``2 * rows * H * (d_h + d_r) * d_model``."""
    d_model = PROJ_D_MODEL.get(w.name)
    if d_model is None or w.dtype != "bf16":
        return None
    T, M = w.B * w.Hq, w.H * (w.d_h + w.d_r)
    t = {k: v.to(device) for k, v in synth.query_tensors(w.seed + 300, w.B, w.Hq, w.H, w.d_h,
                                                          w.d_r, d_model).items()}
    q_nope = torch.empty(w.B, w.Hq, w.H, w.d_h, dtype=torch.bfloat16, device=device)
    q_rope = torch.empty(w.B, w.Hq, w.H, w.d_r, dtype=torch.bfloat16, device=device)
    ws = torch.empty(mla.mla_project_query_workspace_size(w.B, w.Hq, d_model, dims),
                     dtype=torch.uint8, device=device)
    ms = _time_calls(lambda: mla.mla_project_query(t["h"], t["W_Q"], t["W_QR"], dev["seqlens"],
                                                   dims, q_nope, q_rope, ws, stream=stream),
                     max(3, min(args.steps, 50)), flush, stream)
    nbytes = 2 * M * d_model + 2 * T * d_model + 2 * T * M
    flops = 2 * T * M * d_model
    peaks, _ = load_peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {
        "ms": round(ms, 5),
        "d_model": d_model,
        "rows": T,
        "algorithmic_bytes": nbytes,
        "gbs": round(gbs, 1),
        "tflops": round(flops / (ms * 1e-3) / 1e12, 2),
        "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
        "launches": 2,
    }


def measure_o_proj(mla, args, w, out, dims, flush, stream, device):
    """``mla_o_proj`` on the step's head outputs (B * Hq rows of H * d_h) at the
    model's hidden size.  Algorithmic bytes: ``W_O`` once, the head outputs
    in and ``u`` out; FLOPs ``2 * rows * H * d_h * d_model``."""
    d_model = PROJ_D_MODEL.get(w.name)
    if d_model is None or w.dtype != "bf16":
        return None
    T, K = w.B * w.Hq, w.H * w.d_h
    W_O = synth.o_proj_tensors(w.seed + 200, 1, 1, w.H, w.d_h, d_model)["W_O"].to(device)
    u = torch.empty(w.B, w.Hq, d_model, dtype=torch.bfloat16, device=device)
    ws = torch.empty(mla.mla_o_proj_workspace_size(w.B, w.Hq, d_model, dims),
                     dtype=torch.uint8, device=device)
    ms = _time_calls(lambda: mla.mla_o_proj(out, W_O, u, dims, ws, stream=stream),
                     max(3, min(args.steps, 50)), flush, stream)
    nbytes = 2 * d_model * K + 2 * T * K + 2 * T * d_model
    flops = 2 * T * K * d_model
    peaks, _ = load_peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {
        "ms": round(ms, 5),
        "d_model": d_model,
        "rows": T,
        "algorithmic_bytes": nbytes,
        "gbs": round(gbs, 1),
        "tflops": round(flops / (ms * 1e-3) / 1e12, 2),
        "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
        "launches": 2,
    }


# prompts of the prefill measurement: four 4096-token sequences, packed
PREFILL_SEQLENS = [4096] * 4


def measure_prefill(mla, args, w, flush, stream, device):
    """``mla_prefill`` (standard order: K and V rebuilt by one GEMM, then
    causal attention) on four 4096-token prompts with the workload's heads.
    Algorithmic FLOPs: the rebuild ``2 T H (d_h + d_h) d_c`` plus the
    attention's ``2 H (d_h + d_r + d_h)`` per visible (query, key) pair,
    ``T_b (T_b + 1) / 2`` pairs per prompt; both are tensor-core work, so the
    fraction is taken of the measured dense bf16 peak."""
    if w.dtype != "bf16" or (w.d_h, w.d_c, w.d_r) != (128, 512, 64):
        return None
    t = {k: v.to(device) for k, v in synth.prefill_tensors(w.seed + 400, PREFILL_SEQLENS,
                                                            w.H).items()}
    T = sum(PREFILL_SEQLENS)
    dims = mla.Dims(H=w.H, d_h=128, d_c=512, d_r=64, block_size=64, dtype=torch.bfloat16)
    out = torch.empty(T, w.H, 128, dtype=torch.bfloat16, device=device)
    lse = torch.empty(T, w.H, dtype=torch.float32, device=device)
    ws = torch.zeros(mla.mla_prefill_workspace_size(T, dims), dtype=torch.uint8, device=device)
    ms = _time_calls(lambda: mla.mla_prefill(t["q_nope"], t["q_rope"], t["c_kv"], t["k_r"],
                                             t["W_UK"], t["W_UV"], t["cu_seqlens"],
                                             max(PREFILL_SEQLENS), dims, out, lse, ws,
                                             stream=stream),
                     max(3, min(args.steps, 20)), flush, stream)
    kv_flops, attn_flops = prefill_work(PREFILL_SEQLENS, w.H)
    peaks, _ = load_peaks()
    tflops = (kv_flops + attn_flops) / (ms * 1e-3) / 1e12
    return {
        "ms": round(ms, 5),
        "prompts": PREFILL_SEQLENS,
        "H": w.H,
        "kv_rebuild_flops": kv_flops,
        "attention_flops": attn_flops,
        "tflops": round(tflops, 1),
        "tensor_frac_of_burst": round(tflops / peaks["bf16_tflops"], 4),
        "launches": 2,
    }


def measure_project_append(mla, args, w, dev, inp, dims, flush, stream, device):
    """``mla_project_append`` for the step's new tokens (B * Hq of them) at the
    model's hidden size: CUDA events around each call, L2 flushed before it,
    all calls enqueued behind a spin kernel.  The algorithmic bytes are the
    two weights, the hidden states and the cache rows written; the FLOPs
    ``2 * tokens * (d_c + d_r) * d_model``."""
    d_model = PROJ_D_MODEL.get(w.name)
    if d_model is None or w.dtype != "bf16":
        return None
    T = w.B * w.Hq
    pt = {k: v.to(device) for k, v in synth.project_tensors(w.seed + 100, w.B, w.Hq, d_model,
                                                            w.d_c, w.d_r).items()}
    ws = torch.empty(mla.mla_project_append_workspace_size(w.B, w.Hq, d_model, dims),
                     dtype=torch.uint8, device=device)

    def call():
        mla.mla_project_append(pt["h"], pt["W_DKV"], pt["W_KR"], dev["cache"],
                               inp["num_blocks"], dev["block_table"], dev["seqlens"], dims, ws,
                               stream=stream)

    ms = _time_calls(call, max(3, min(args.steps, 50)), flush, stream)
    D = w.d_c + w.d_r
    nbytes = 2 * D * d_model + 2 * T * d_model + 2 * T * D
    flops = 2 * T * D * d_model
    peaks, _ = load_peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {
        "ms": round(ms, 5),
        "d_model": d_model,
        "tokens": T,
        "algorithmic_bytes": nbytes,
        "gbs": round(gbs, 1),
        "tflops": round(flops / (ms * 1e-3) / 1e12, 2),
        "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
        "launches": 2,
    }


def smi_index(local_index):
    """nvidia-smi's name for a CUDA device index (honours CUDA_VISIBLE_DEVICES)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local_index < len(ids):
            return ids[local_index]
    return str(local_index)


def decode_launches(mla, dims, w):
    """Kernels one mla_decode call launches on this path."""
    return 2


def load_traffic(name):
    """DRAM bytes of the decode kernel from the committed ncu summary, when it
    was captured on the current kernel version (else null)."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(name)
    return e if e else None


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline, and the reference arm)
# ---------------------------------------------------------------------------


def oracle_cores():
    try:
        from threadpoolctl import threadpool_info
        n = [p["num_threads"] for p in threadpool_info() if p.get("internal_api") == "openblas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


def time_oracle_sample(name, budget_s, heads_per_chunk=8, inputs=None):
    """Run the fp64 oracle on (sequence, head) rows of the workload until
    ``budget_s`` seconds have passed; returns (algorithmic flops, seconds,
    description)."""
    from oracle import mla as omla

    w = synth.WORKLOADS[name]
    if inputs is None:
        inputs = synth.make_bf16_inputs(name)
    W_UK = inputs["W_UK"].double().numpy()
    W_UV = inputs["W_UV"].double().numpy()
    bs = w.block_size
    flops = 0
    rows = 0
    t0 = time.perf_counter()
    b = 0
    done = False
    while not done:
        n = int(inputs["seqlens"][b])
        nblk = -(-n // bs)
        cache = inputs["cache"][inputs["block_table"][b, :nblk].long()].double().numpy()
        table = np.arange(nblk)[None, :]
        for h0 in range(0, w.H, heads_per_chunk):
            hs = list(range(h0, min(w.H, h0 + heads_per_chunk)))
            omla.mla_decode(inputs["q_nope"][b:b + 1].double().numpy(),
                            inputs["q_rope"][b:b + 1].double().numpy(), cache, table,
                            inputs["seqlens"][b:b + 1].numpy(), W_UK, W_UV, w.Hq,
                            head_indices=hs)
            vt = visible_tokens([n], w.Hq)
            flops += len(hs) * (2 * (w.d_c + w.d_r) + 2 * w.d_c) * vt
            rows += len(hs) * w.Hq
            if time.perf_counter() - t0 >= budget_s:
                done = True
                break
        b = (b + 1) % w.B
    dt = time.perf_counter() - t0
    return flops, dt, f"{rows} (sequence, head) rows of the {name} workload"


def run_reference(args, rank):
    if rank != 0:
        return None
    w = synth.WORKLOADS[args.workload]
    inputs = synth.make_bf16_inputs(args.workload)
    times, flops_all = [], []
    desc = ""
    for it in range(args.warmup + args.steps):
        fl, dt, desc = time_oracle_sample(args.workload, args.ref_step_s, inputs=inputs)
        if it >= args.warmup:
            times.append(dt)
            flops_all.append(fl)
    value = sum(flops_all) / sum(times) / 1e12
    cores = oracle_cores()
    return {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "impl": "reference",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * float(np.mean(times)), 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": synth.DESCRIPTIONS[args.workload], "name": args.workload},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: {desc} (~{args.ref_step_s:.0f} s of fp64 "
                                   f"un-absorbed oracle on the host)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_decode_only(args, device):
    """``--decode-only``: ``mla_decode`` alone on the chosen workload (for
    profiling one workload's decode kernel), same timing and roofline as the
    ``configs`` record of the full run."""
    import mla_latent_kv_74_b300 as mla
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    res = measure_other_configs(mla, argparse.Namespace(workload=None, steps=args.steps),
                                flush, stream, device, names=(args.workload,), batch=args.batch)
    r = res[args.workload]
    return {"metric": "mla_decode time, fraction of max(bytes/HBM, FLOPs/bf16 peak)",
            "value": r["roofline_time_frac"], "unit": "fraction", "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic", "decode": r}


def run_prefill_only(args, device):
    """``--prefill-only``: the prefill measurement alone (for profiling it)."""
    import mla_latent_kv_74_b300 as mla
    w = synth.WORKLOADS[args.workload]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    res = measure_prefill(mla, args, w, flush, stream, device)
    if res is None:
        return {"prefill": None, "why": f"no prefill path for the {w.name} workload's dims"}
    return {"metric": "MLA prefill tensor TFLOP/s (K/V rebuild + causal attention)",
            "value": res["tflops"], "unit": "TFLOP/s", "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic", "prefill": res}


# ---------------------------------------------------------------------------


def spawn_ranks(n, cmd=None):
    """Run ``n`` ranks of this benchmark on this node, one process per GPU,
    when it was started without torchrun: child r gets RANK = LOCAL_RANK = r,
    WORLD_SIZE = n and a rendezvous on 127.0.0.1.  ``cmd`` (default: this
    script with the same arguments) is the child command line.  Returns the
    first non-zero exit code of the children, else 0."""
    import socket

    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    if cmd is None:
        cmd = [sys.executable, os.path.abspath(__file__), *sys.argv[1:]]
    procs = []
    for r in range(n):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(n),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen(cmd, env=env))
    rc = 0
    for proc in procs:
        code = proc.wait()
        rc = rc or code
    return rc


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="v2", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch size (small profiling captures)")
    ap.add_argument("--cpu-baseline-s", type=float, default=15.0,
                    help="seconds of oracle work for the cpu_baseline key (0 = skip)")
    ap.add_argument("--ref-step-s", type=float, default=3.0,
                    help="seconds of oracle work per step of the reference arm")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time only mla_prefill (four 4096-token prompts) and print its line")
    ap.add_argument("--decode-only", action="store_true",
                    help="time only mla_decode on --workload and print its line")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # not under torchrun: one process per GPU, started here
        sys.exit(spawn_ranks(args.gpus))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        res = run_reference(args, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return

    if args.decode_only:
        if rank == 0:
            device = torch.device("cuda", local_rank)
            torch.cuda.set_device(device)
            print(json.dumps(run_decode_only(args, device)), flush=True)
        return

    if args.prefill_only:
        if rank == 0:
            device = torch.device("cuda", local_rank)
            torch.cuda.set_device(device)
            print(json.dumps(run_prefill_only(args, device)), flush=True)
        return

    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    res = run_ours(args, rank, world, device)
    if res is not None:
        if args.cpu_baseline_s > 0:
            fl, dt, desc = time_oracle_sample(args.workload, args.cpu_baseline_s)
            res["cpu_baseline"] = {
                "value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": oracle_cores(),
                "kind": "oracle",
                "sample": f"{desc}; {dt:.1f} s of the fp64 un-absorbed oracle on the host",
            }
        else:
            res["cpu_baseline"] = None
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
