"""Build ``libmla.so`` (the C-ABI library) in-tree with nvcc for sm_103a.

    python mla_latent_kv_74_b300/build.py                  # build if sources changed
    python mla_latent_kv_74_b300/build.py --force          # always rebuild
    python mla_latent_kv_74_b300/build.py --verbose-ptxas  # print -Xptxas -v
    python mla_latent_kv_74_b300/build.py --trace          # developer build with
                                                           # per-tile decode timestamps

(Run it by path: the package's __init__ loads the library this script builds.)

Each ``csrc/*.cu`` compiles to an object under ``_build/`` (in parallel) and
the objects link into ``mla_latent_kv_74_b300/libmla.so``.  No GPU is needed:
nvcc cross-compiles.
"""

from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmla.so")
TRACE_LIB = os.path.join(BUILD, "trace", "libmla_trace.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include")]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh"))
            + [os.path.join(ROOT, "include", "mla.h"), __file__])


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src, verbose_ptxas, out_dir=BUILD, defines=()):
    obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [NVCC, *ARCH, *FLAGS, *("-D" + d for d in defines), "-c", src, "-o", obj]
    if verbose_ptxas:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, (r.stdout + r.stderr)


def build(force: bool = False, verbose_ptxas: bool = False, quiet: bool = True,
          trace: bool = False) -> str:
    """Compile every CUDA source and link ``libmla.so``; returns its path.

    ``trace=True`` builds the developer variant ``_build/trace/libmla_trace.so``
    instead (MLA_TRACE: the decode kernel records per-tile timestamps that
    ``mla_debug_read_trace`` copies out); the package never loads it."""
    lib = TRACE_LIB if trace else LIB
    out_dir = os.path.dirname(TRACE_LIB) if trace else BUILD
    defines = ("MLA_TRACE",) if trace else ()
    if not force and not verbose_ptxas and not _stale(lib, _deps()):
        return lib
    os.makedirs(out_dir, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose_ptxas, out_dir, defines), srcs))
    objs = [o for o, _ in results]
    if verbose_ptxas or not quiet:
        for _, log in results:
            if log.strip():
                print(log, file=sys.stderr)
    tmp = lib + ".tmp"
    cmd = [NVCC, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-ldl", "-lrt",
           "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true")
    ap.add_argument("--trace", action="store_true")
    args = ap.parse_args()
    print(build(force=args.force, verbose_ptxas=args.verbose_ptxas, quiet=False,
                trace=args.trace))
