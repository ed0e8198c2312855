"""Build libfp8q.so (the sm_103a CUDA library) in-tree with nvcc.

Each translation unit under csrc/ is compiled in parallel for
``-gencode arch=compute_103a,code=sm_103a`` and linked into
``quantize_fp8_gemm_gb300/libfp8q.so``, which exports the plain C ABI of
include/fp8q.h (and the hooks of include/fp8q_testing.h).  The measured
comparators under csrc/comparators/ (the unfused three-pass quantize,
include/fp8q_naive.h) go into a library of their own, libfp8q_naive.so, so
the product library holds only the path.  No CMake, no torch extension
machinery.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfp8q.so")
NAIVE_LIB = os.path.join(PKG, "libfp8q_naive.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-fno-strict-aliasing",
              "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfp8q.so")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def comparator_sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "comparators", "*.cu")))


def _deps() -> list[str]:
    return (sources() + comparator_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) +
            glob.glob(os.path.join(ROOT, "include", "*.h")))


def up_to_date() -> bool:
    if not (os.path.exists(LIB) and os.path.exists(NAIVE_LIB)):
        return False
    t = min(os.path.getmtime(LIB), os.path.getmtime(NAIVE_LIB))
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link libfp8q.so and libfp8q_naive.so if any source is newer;
    return the path of libfp8q.so."""
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src: str) -> tuple[str, str]:
        sub = "comparators_" if os.path.dirname(src).endswith("comparators") else ""
        obj = os.path.join(BUILD, sub + os.path.basename(src) + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    srcs = sources()
    csrcs = comparator_sources()
    with ThreadPoolExecutor(max(1, min(len(srcs) + len(csrcs), os.cpu_count() or 4))) as ex:
        results = list(ex.map(compile_one, srcs + csrcs))
    if verbose or ptxas_info:
        for _, log in results:
            if log.strip():
                print(log, file=sys.stderr)
    for lib, objs in ((LIB, [o for o, _ in results[:len(srcs)]]), (NAIVE_LIB, [o for o, _ in results[len(srcs):]])):
        tmp = lib + ".tmp"
        cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of {os.path.basename(lib)} failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
