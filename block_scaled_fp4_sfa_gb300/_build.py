"""Builds the CUDA library (libfp4gemm.so) in-tree with nvcc for sm_103a.

Three translation units (the tcgen05 GEMM, the narrow-M kernel and the
quantiser) compiled in parallel, one -gencode, then linked into one shared
library; the static CUDA runtime is linked in and the driver's tensor-map
encoder is looked up at run time, so the library needs no -lcuda.
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
SOURCES = [os.path.join(CSRC, "fp4_gemm.cu"), os.path.join(CSRC, "fp4_quant.cu"), os.path.join(CSRC, "fp4_gemv.cu")]
DEPS = SOURCES + [os.path.join(CSRC, "ptx.cuh"), os.path.join(CSRC, "epilogue.cuh"), os.path.join(CSRC, "fp4_gemv.cuh"),
                  os.path.join(INCLUDE, "fp4_gemm.h"),
                  os.path.join(INCLUDE, "fp4_quant.h")]

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
    objs = [tmp + ".%d.o" % i for i in range(len(SOURCES))]
    procs = []
    for src, obj in zip(SOURCES, objs):
        cmd = [nvcc(), *flags(extra), "-c", "-o", obj, src]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((cmd, subprocess.Popen(cmd)))
    failed = [cmd for cmd, p in procs if p.wait() != 0]
    try:
        if failed:
            raise subprocess.CalledProcessError(1, failed[0])
        subprocess.run([nvcc(), ARCH, "-shared", "-o", tmp, *objs], check=True)
    finally:
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True,
          extra=("-Xptxas", "-v") if "--ptxas-v" in sys.argv else ())
