"""Build libfa.so (and the test-only primitive library) with nvcc for sm_103a.

Each .cu translation unit compiles in parallel to an object file under
`_build/`, then nvcc links the shared library next to this file. Nothing is
installed; the library stays in-tree.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(ROOT, "_build")

LIB_SOURCES = ["fa_api.cu", "fa_prefill.cu", "fa_decode.cu", "fa_backward.cu"]
SELFTEST_SOURCES = ["fa_selftest.cu"]
LIB_NAME = "libfa.so"
SELFTEST_NAME = "libfa_selftest.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libfa.so")
    return cand


def _compile(src: str, extra=()) -> str:
    os.makedirs(BUILD, exist_ok=True)
    obj = os.path.join(BUILD, os.path.basename(src).replace(".cu", ".o"))
    cmd = [_nvcc(), *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    return obj


def _link(objs, out):
    cmd = [_nvcc(), *ARCH, "-shared", "-cudart", "shared", "-Xlinker", "-rpath", "-Xlinker",
           "/usr/local/cuda/lib64", *objs, "-o", out]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")


def build(verbose_ptxas: bool = False, selftest: bool = True) -> str:
    """Compile and link; returns the path of libfa.so."""
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    srcs = LIB_SOURCES + (SELFTEST_SOURCES if selftest else [])
    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = dict(zip(srcs, ex.map(lambda s: _compile(s, extra), srcs)))
    lib = os.path.join(HERE, LIB_NAME)
    _link([objs[s] for s in LIB_SOURCES], lib)
    if selftest:
        _link([objs[s] for s in SELFTEST_SOURCES], os.path.join(HERE, SELFTEST_NAME))
    return lib


if __name__ == "__main__":
    print(build(verbose_ptxas="-v" in sys.argv))
