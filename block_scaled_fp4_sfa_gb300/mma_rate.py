"""Builds and runs the MMA issue-rate micro-benchmark (csrc/mma_rate.cu).

    python -m block_scaled_fp4_sfa_gb300.mma_rate

It measures, on every SM at once, how many cycles a k-tile of dense
block-scaled FP4 MMAs (four K = 64 `tcgen05.mma`) takes when nothing else
limits the issuing thread: the tensor pipe's own rate, which bounds the GEMM
kernel's main loop, and what staging scales through `tcgen05.cp` in the same
thread or a commit per k-tile adds. Needs a GPU; the binary is built in-tree.
"""
from __future__ import annotations

import os
import subprocess
import sys

from . import _build

SRC = os.path.join(_build.CSRC, "mma_rate.cu")
EXE = os.path.join(_build.PKG, "mma_rate_bench")


def build() -> str:
    if not os.path.exists(EXE) or os.path.getmtime(EXE) < max(os.path.getmtime(SRC),
                                                            os.path.getmtime(os.path.join(_build.CSRC, "ptx.cuh"))):
        subprocess.run([_build.nvcc(), _build.ARCH, "-O3", "-std=c++17", "--expt-relaxed-constexpr", "-I", _build.CSRC,
                        "-o", EXE, SRC], check=True)
    return EXE


if __name__ == "__main__":
    sys.exit(subprocess.run([build()]).returncode)
