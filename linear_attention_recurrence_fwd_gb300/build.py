"""Build libkda.so (the product library) and libkda_probe.so (test-only
layout probes) in-tree with nvcc for sm_103a.

Each translation unit compiles in its own process (in parallel), then one
shared-library link.  Rebuilds only when a source or header is newer than
the library.  Usage: ``python -m linear_attention_recurrence_fwd_gb300.build``.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libkda.so")
PROBE_LIB = os.path.join(PKG, "libkda_probe.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]

PRODUCT_SOURCES = ["kda_api.cu", "kda_decode.cu", "kda_chunk.cu", "kda_bwd.cu", "kda_host.cu"]
PROBE_SOURCES = ["kda_probe.cu"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or install the CUDA toolkit)")


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
                   "-I", os.path.join(ROOT, "include"), "-I", CSRC, *extra]


def _deps():
    return (glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(ROOT, "include", "*.h"))
            + [os.path.abspath(__file__)])


def _stale(target: str) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in _deps())


def _compile(src: str, extra=()) -> str:
    os.makedirs(OBJ, exist_ok=True)
    obj = os.path.join(OBJ, os.path.basename(src) + ".o")
    cmd = [nvcc(), *_flags(extra), "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def _link(objs, out):
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed for {out}:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> list[str]:
    """Compile both libraries if stale; returns their paths."""
    jobs = []
    if force or _stale(LIB):
        jobs.append((LIB, PRODUCT_SOURCES))
    if force or _stale(PROBE_LIB):
        jobs.append((PROBE_LIB, PROBE_SOURCES))
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if jobs:
        srcs = sorted({s for _, group in jobs for s in group})
        with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
            objs = dict(zip(srcs, ex.map(lambda s: _compile(s, extra), srcs)))
        for out, group in jobs:
            _link([objs[s] for s in group], out)
            if verbose:
                print("built", out, file=sys.stderr)
    return [LIB, PROBE_LIB]


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas-info" in sys.argv)
