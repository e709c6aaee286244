"""Seeded synthetic inputs shared by the oracle-side tests and the CUDA path.

This module only draws random numbers and lays out the paged cache; it holds
none of the method's arithmetic.  Both sides (``oracle/`` and the CUDA
library) consume exactly the tensors produced here.

Workloads (shapes of the DeepSeek-V2 family: H=128, d_h=128, d_c=512, d_r=64):

=========  =====  ====  ==========================  ==  ====  ==========
name       H      B     seqlens                     Hq  seed  dtype
=========  =====  ====  ==========================  ==  ====  ==========
tiny       4      1     32                          1   0     fp32
lite       16     32    4096                        1   1     bf16
v2         128    64    8192                        1   2     bf16
mtp        128    128   uniform integers [256,32768] 2  3     bf16
long       128    4     131072                      1   4     bf16
=========  =====  ====  ==========================  ==  ====  ==========

Value recipe (bf16 workloads): ``c_KV, k_R, q_nope, q_rope ~ N(0, 1)``,
``W_UK, W_UV ~ N(0, 1/512)``; drawn in fp32 from ``torch.Generator`` on the
CPU and rounded to bf16 (round-to-nearest-even).  The block table of every
paged workload is a seeded random permutation of exactly
``sum_b ceil(seqlen_b / 64)`` physical blocks; unused table entries are -1.

The tiny fp32 workload is specified by hidden states and weights
(``h ~ N(0,1)``, every weight ``~ N(0,1)/sqrt(fan_in)``, ``d_model = 64``);
its cache rows and queries are derived from them by the test harness.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

BLOCK_SIZE = 64


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    H: int
    d_h: int
    d_c: int
    d_r: int
    B: int
    Hq: int
    seed: int
    dtype: str  # "bf16" or "fp32"
    seqlen: Optional[int] = None  # fixed length, or None for ragged
    seqlen_range: Optional[tuple] = None  # inclusive range for ragged lengths
    block_size: int = BLOCK_SIZE
    d_model: int = 0  # tiny workload only

    @property
    def D(self) -> int:
        return self.d_c + self.d_r


WORKLOADS = {
    "tiny": Workload("tiny", H=4, d_h=16, d_c=16, d_r=8, B=1, Hq=1, seed=0,
                     dtype="fp32", seqlen=32, d_model=64),
    "lite": Workload("lite", H=16, d_h=128, d_c=512, d_r=64, B=32, Hq=1, seed=1,
                     dtype="bf16", seqlen=4096),
    "v2": Workload("v2", H=128, d_h=128, d_c=512, d_r=64, B=64, Hq=1, seed=2,
                   dtype="bf16", seqlen=8192),
    "mtp": Workload("mtp", H=128, d_h=128, d_c=512, d_r=64, B=128, Hq=2, seed=3,
                    dtype="bf16", seqlen_range=(256, 32768)),
    "long": Workload("long", H=128, d_h=128, d_c=512, d_r=64, B=4, Hq=1, seed=4,
                     dtype="bf16", seqlen=131072),
}

DESCRIPTIONS = {
    "tiny": "tiny fp32 MLA decode: d_model=64, H=4, d_h=16, d_r=8, d_c=16, B=1, seqlen=32, Hq=1",
    "lite": "DeepSeek-V2-Lite-shaped bf16 decode: H=16, d_h=128, d_r=64, d_c=512, B=32, seqlen=4096, Hq=1, paged block 64",
    "v2": "DeepSeek-V2-shaped bf16 decode: H=128, d_h=128, d_r=64, d_c=512, B=64, seqlen=8192, Hq=1, paged block 64, permuted block_table",
    "mtp": "ragged MTP-style bf16 decode: H=128, d_h=128, d_r=64, d_c=512, B=128, seqlens U[256,32768], Hq=2 causal, paged block 64",
    "long": "long-context bf16 decode: H=128, d_h=128, d_r=64, d_c=512, B=4, seqlen=131072, Hq=1, paged block 64",
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _normal(g, shape, std=1.0, dtype=torch.bfloat16):
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def draw_seqlens(w: Workload, g: torch.Generator) -> np.ndarray:
    if w.seqlen is not None:
        return np.full(w.B, w.seqlen, dtype=np.int32)
    lo, hi = w.seqlen_range
    s = torch.randint(lo, hi + 1, (w.B,), generator=g, dtype=torch.int64)
    return s.numpy().astype(np.int32)


def paged_block_table(seqlens: np.ndarray, block_size: int, g: torch.Generator):
    """A random permutation of exactly ``sum ceil(seqlen/bs)`` physical blocks,
    dealt out to the sequences in order.  Returns ``(table [B, max_blocks]
    int32 with -1 padding, num_blocks)``."""
    nblk = [(int(s) + block_size - 1) // block_size for s in seqlens]
    total = sum(nblk)
    perm = torch.randperm(total, generator=g).numpy().astype(np.int32)
    max_blocks = max(nblk) if nblk else 0
    table = np.full((len(seqlens), max(max_blocks, 1)), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[off:off + n]
        off += n
    return table, total


def make_bf16_inputs(name: str, seqlens_override=None, B_override=None):
    """Every input of one decode step of a bf16 workload, on the CPU.

    Returns a dict of torch tensors:

    ``cache``       [num_blocks, 64, d_c + d_r] bf16 -- state before the append
    ``c_kv_new``    [B, Hq, d_c] bf16 -- latents of the Hq current tokens
    ``k_r_new``     [B, Hq, d_r] bf16 -- their (already rotated) RoPE keys
    ``q_nope``      [B, Hq, H, d_h] bf16
    ``q_rope``      [B, Hq, H, d_r] bf16 (already rotated)
    ``W_UK, W_UV``  [H, d_h, d_c] bf16
    ``block_table`` [B, max_blocks] int32
    ``seqlens``     [B] int32 -- lengths after the append
    """
    w = WORKLOADS[name]
    if B_override is not None:
        w = dataclasses.replace(w, B=B_override)
    g = _gen(w.seed)
    if seqlens_override is not None:
        seqlens = np.asarray(seqlens_override, dtype=np.int32)
        w = dataclasses.replace(w, B=len(seqlens))
    else:
        seqlens = draw_seqlens(w, g)
    table, num_blocks = paged_block_table(seqlens, w.block_size, g)
    D = w.D
    cache = _normal(g, (num_blocks, w.block_size, D))
    c_kv_new = _normal(g, (w.B, w.Hq, w.d_c))
    k_r_new = _normal(g, (w.B, w.Hq, w.d_r))
    q_nope = _normal(g, (w.B, w.Hq, w.H, w.d_h))
    q_rope = _normal(g, (w.B, w.Hq, w.H, w.d_r))
    wstd = 1.0 / math.sqrt(w.d_c)
    W_UK = _normal(g, (w.H, w.d_h, w.d_c), std=wstd)
    W_UV = _normal(g, (w.H, w.d_h, w.d_c), std=wstd)
    return {
        "workload": w,
        "cache": cache,
        "c_kv_new": c_kv_new,
        "k_r_new": k_r_new,
        "q_nope": q_nope,
        "q_rope": q_rope,
        "W_UK": W_UK,
        "W_UV": W_UV,
        "block_table": torch.from_numpy(table),
        "seqlens": torch.from_numpy(seqlens),
        "num_blocks": num_blocks,
    }


def make_tiny_raw(seed: int = 0):
    """Hidden states and weights of the tiny fp32 workload (fp64 numpy).

    ``h [32, 64] ~ N(0,1)``; ``W_DKV [16, 64]``, ``W_KR [8, 64]``,
    ``W_Q [64, 64]``, ``W_QR [32, 64]`` each ``~ N(0,1)/sqrt(64)``;
    ``W_UK, W_UV [4, 16, 16] ~ N(0,1)/sqrt(16)`` (fan-in is the latent width).
    """
    w = WORKLOADS["tiny"]
    g = _gen(seed)
    d = w.d_model

    def draw(shape, fan_in=None):
        x = torch.randn(shape, generator=g, dtype=torch.float64)
        if fan_in is not None:
            x = x / math.sqrt(fan_in)
        return x.numpy()

    return {
        "workload": w,
        "h": draw((w.seqlen, d)),
        "W_DKV": draw((w.d_c, d), d),
        "W_KR": draw((w.d_r, d), d),
        "W_Q": draw((w.H * w.d_h, d), d),
        "W_QR": draw((w.H * w.d_r, d), d),
        "W_UK": draw((w.H, w.d_h, w.d_c), w.d_c),
        "W_UV": draw((w.H, w.d_h, w.d_c), w.d_c),
    }


def random_small(seed, H, d_h, d_c, d_r, seqlens, Hq, block_size=BLOCK_SIZE,
                 dtype=torch.bfloat16, permute=True):
    """Small random decode inputs of arbitrary shape for parity sweeps.

    Same value recipe as the bf16 workloads; ``dtype`` may be fp32.
    """
    g = _gen(seed)
    seqlens = np.asarray(seqlens, dtype=np.int32)
    B = len(seqlens)
    if permute:
        table, num_blocks = paged_block_table(seqlens, block_size, g)
    else:
        nblk = [(int(s) + block_size - 1) // block_size for s in seqlens]
        num_blocks = sum(nblk)
        table = np.full((B, max(max(nblk), 1)), -1, dtype=np.int32)
        off = 0
        for b, n in enumerate(nblk):
            table[b, :n] = np.arange(off, off + n)
            off += n
    num_blocks = max(num_blocks, 1)
    D = d_c + d_r
    wstd = 1.0 / math.sqrt(d_c)
    return {
        "cache": _normal(g, (num_blocks, block_size, D), dtype=dtype),
        "c_kv_new": _normal(g, (B, Hq, d_c), dtype=dtype),
        "k_r_new": _normal(g, (B, Hq, d_r), dtype=dtype),
        "q_nope": _normal(g, (B, Hq, H, d_h), dtype=dtype),
        "q_rope": _normal(g, (B, Hq, H, d_r), dtype=dtype),
        "W_UK": _normal(g, (H, d_h, d_c), std=wstd, dtype=dtype),
        "W_UV": _normal(g, (H, d_h, d_c), std=wstd, dtype=dtype),
        "block_table": torch.from_numpy(table),
        "seqlens": torch.from_numpy(seqlens),
        "num_blocks": num_blocks,
    }


def project_inputs(seed, seqlens, n_new, d_model, d_c=512, d_r=64, block_size=BLOCK_SIZE):
    """Inputs of the fused projection-and-append step: hidden states of the
    ``n_new`` newest tokens ``h ~ N(0,1)`` [B, n_new, d_model], weights
    ``W_DKV`` [d_c, d_model] and ``W_KR`` [d_r, d_model] ``~ N(0, 1/d_model)``
    (so the projected values have unit variance), and a paged cache filled
    with N(0,1) rows that the step must overwrite only where it writes.
    All bf16."""
    g = _gen(seed)
    seqlens = np.asarray(seqlens, dtype=np.int32)
    B = len(seqlens)
    table, num_blocks = paged_block_table(np.maximum(seqlens, 1), block_size, g)
    out = project_tensors(g, B, n_new, d_model, d_c, d_r)
    out.update({
        "cache": _normal(g, (num_blocks, block_size, d_c + d_r)),
        "block_table": torch.from_numpy(table),
        "seqlens": torch.from_numpy(seqlens),
        "num_blocks": num_blocks,
    })
    return out


def project_tensors(g, B, n_new, d_model, d_c=512, d_r=64):
    """``h``, ``W_DKV``, ``W_KR`` of the projection step, drawn from ``g``
    (a seed or a ``torch.Generator``) with the recipe of ``project_inputs``."""
    if not isinstance(g, torch.Generator):
        g = _gen(g)
    wstd = 1.0 / math.sqrt(d_model)
    return {
        "h": _normal(g, (B, n_new, d_model)),
        "W_DKV": _normal(g, (d_c, d_model), std=wstd),
        "W_KR": _normal(g, (d_r, d_model), std=wstd),
    }


def o_proj_tensors(seed, B, Hq, H, d_h, d_model):
    """Inputs of the output projection: head outputs ``out ~ N(0,1)``
    [B, Hq, H, d_h] and ``W_O ~ N(0, 1/(H*d_h))`` [d_model, H*d_h] (so ``u``
    has unit variance).  bf16."""
    g = _gen(seed)
    return {
        "out": _normal(g, (B, Hq, H, d_h)),
        "W_O": _normal(g, (d_model, H * d_h), std=1.0 / math.sqrt(H * d_h)),
    }


def query_tensors(seed, B, Hq, H, d_h, d_r, d_model):
    """Inputs of the query projections: ``h ~ N(0,1)`` [B, Hq, d_model] and
    ``W_Q`` [H*d_h, d_model], ``W_QR`` [H*d_r, d_model] ``~ N(0, 1/d_model)``.
    bf16."""
    g = _gen(seed)
    wstd = 1.0 / math.sqrt(d_model)
    return {
        "h": _normal(g, (B, Hq, d_model)),
        "W_Q": _normal(g, (H * d_h, d_model), std=wstd),
        "W_QR": _normal(g, (H * d_r, d_model), std=wstd),
    }


def prefill_tensors(seed, seqlens, H, d_h=128, d_c=512, d_r=64):
    """Inputs of a packed prefill: sequences of the given lengths laid end to
    end (``cu_seqlens`` [B+1] int32, the prefix sums), ``q_nope [T, H, d_h]``,
    ``q_rope [T, H, d_r]``, ``c_kv [T, d_c]``, ``k_r [T, d_r]`` ``~ N(0,1)``
    and ``W_UK, W_UV [H, d_h, d_c] ~ N(0, 1/d_c)`` (the decode recipe, so
    scaled scores have unit variance).  bf16."""
    g = _gen(seed)
    cu = np.zeros(len(seqlens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(seqlens, dtype=np.int64))
    T = int(cu[-1])
    wstd = 1.0 / math.sqrt(d_c)
    return {
        "cu_seqlens": torch.from_numpy(cu),
        "q_nope": _normal(g, (T, H, d_h)),
        "q_rope": _normal(g, (T, H, d_r)),
        "c_kv": _normal(g, (T, d_c)),
        "k_r": _normal(g, (T, d_r)),
        "W_UK": _normal(g, (H, d_h, d_c), std=wstd),
        "W_UV": _normal(g, (H, d_h, d_c), std=wstd),
    }
