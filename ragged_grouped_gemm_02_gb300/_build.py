"""Build librgg.so (the C-ABI CUDA library) in-tree with nvcc for sm_103a.

Each translation unit in csrc/ is compiled in parallel, then linked into
``ragged_grouped_gemm_02_gb300/librgg.so`` with the CUDA runtime linked
statically, so the library needs no libcudart at load time and reaches the
driver only through the runtime's own entry points.

The same sources built with ``-DRGG_DEBUG_CHECKS`` give
``librgg_debug.so``: the same C ABI whose kernels check every copy, store,
TMEM load and tile descriptor against its bounds before issuing it and
report RGG_ERR_DEVICE_BOUNDS instead (csrc/rgg_checks.cuh).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "librgg.so")
LIB_DEBUG = os.path.join(PKG, "librgg_debug.so")

SOURCES = ["rgg_api.cu", "rgg_aux.cu", "rgg_gemm_bm128.cu", "rgg_gemm_bm64.cu", "rgg_gemm_pair.cu",
           "rgg_noalloc.cu", "rgg_gemm_swiglu.cu", "rgg_gemm_fp8.cu", "rgg_gemm_gather.cu",
           "rgg_gemm_mixed.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build librgg.so")


def _inputs_mtime() -> float:
    names = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "rgg.h"), __file__]
    return max(os.path.getmtime(p) for p in names)


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile and link librgg.so and librgg_debug.so if any source is newer
    than them; return the path of librgg.so."""
    stale = [lib for lib in (LIB, LIB_DEBUG) if force or not os.path.exists(lib) or
             os.path.getmtime(lib) < _inputs_mtime()]
    if not stale:
        return LIB
    nvcc = _nvcc()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    if ptxas_verbose:
        common += ["-Xptxas", "-v"]
    jobs = []
    for lib in stale:
        debug = lib == LIB_DEBUG
        out_dir = BUILD + ("_debug" if debug else "")
        os.makedirs(out_dir, exist_ok=True)
        jobs += [(lib, src, out_dir, ["-DRGG_DEBUG_CHECKS"] if debug else []) for src in SOURCES]

    def compile_one(job) -> str:
        _, src, out_dir, extra = job
        obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc] + common + extra + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
        if verbose or ptxas_verbose:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 8)) as ex:
        objs = list(ex.map(compile_one, jobs))
    for lib in stale:
        lib_objs = [o for o, job in zip(objs, jobs) if job[0] == lib]
        tmp = lib + ".tmp%d" % os.getpid()
        cmd = [nvcc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + lib_objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv))
