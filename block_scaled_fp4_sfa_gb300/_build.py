"""Builds the CUDA library (libfp4gemm.so) in-tree with nvcc for sm_103a.

One translation unit, one -gencode; the static CUDA runtime is linked in and
the driver's tensor-map encoder is looked up at run time, so the library needs
no -lcuda.
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libfp4gemm.so")
SOURCES = [os.path.join(CSRC, "fp4_gemm.cu")]
DEPS = SOURCES + [os.path.join(CSRC, "ptx.cuh"), os.path.join(INCLUDE, "fp4_gemm.h")]

ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def flags(extra=()) -> list[str]:
    return [ARCH, "-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC,
            "-Xcompiler", "-fPIC,-O2", *extra]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    """Compile SOURCES into LIB (skipped when LIB is newer than every source)."""
    if not force and up_to_date() and not extra:
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [nvcc(), *flags(extra), "-shared", "-o", tmp, *SOURCES]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True,
          extra=("-Xptxas", "-v") if "--ptxas-v" in sys.argv else ())
