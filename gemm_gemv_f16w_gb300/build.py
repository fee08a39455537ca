"""Builds liblq.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked; a rebuild happens
only when a source or header is newer than the library. No cmake.

build(debug_bounds=True) builds liblq_debug.so instead: the same sources with
LQ_DEBUG_BOUNDS defined, so that every kernel checks its computed global
indices and reports a failed check as LQ_ERR_BOUNDS (no trap). The binding
loads it when LQ_LIBRARY=debug is set in the environment.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "liblq.so")
DEBUG_BUILD = os.path.join(PKG, "_build_debug")
DEBUG_LIB = os.path.join(PKG, "liblq_debug.so")

CUDA_SOURCES = ["lq_api.cu", "lq_gemv.cu", "lq_gemv_chain.cu", "lq_gemv_batch.cu", "lq_argmax.cu", "lq_topk.cu", "lq_gemm.cu", "lq_gemm_tma.cu",
                "lq_noalloc.cu", "lq_gemm_small.cu"]
CXX_SOURCES = ["lq_pack.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(ROOT, "include", "lq.h"))
    files.append(os.path.abspath(__file__))
    return files


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _deps())


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"build failed: {' '.join(cmd)}\n{r.stdout}")
    return r.stdout


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          debug_bounds: bool = False) -> str:
    """Compile and link liblq.so (liblq_debug.so with debug_bounds) if stale;
    returns its path."""
    lib, bdir = (DEBUG_LIB, DEBUG_BUILD) if debug_bounds else (LIB, BUILD)
    if not force and not _stale(lib):
        return lib
    os.makedirs(bdir, exist_ok=True)
    nvcc = _nvcc()
    inc = ["-I", os.path.join(ROOT, "include")]
    defs = ["-DLQ_DEBUG_BOUNDS"] if debug_bounds else []
    jobs = []
    for src in CUDA_SOURCES:
        obj = os.path.join(bdir, src + ".o")
        cmd = [nvcc, *ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
               "-Xcompiler", "-ffp-contract=off", *defs, *inc, "-c", os.path.join(CSRC, src), "-o", obj]
        if ptxas_info:
            cmd.insert(1, "-Xptxas=-v")
        jobs.append((cmd, obj))
    for src in CXX_SOURCES:
        obj = os.path.join(bdir, src + ".o")
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-ffp-contract=off", *inc, "-c",
               os.path.join(CSRC, src), "-o", obj]
        jobs.append((cmd, obj))
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        outs = list(ex.map(lambda j: _run(j[0]), jobs))
    if verbose:
        for o in outs:
            if o.strip():
                print(o)
    tmp = lib + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-o", tmp, *[o for _, o in jobs], "-lpthread"])
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                debug_bounds="--debug-bounds" in sys.argv))
