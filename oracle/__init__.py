"""CPU oracle for the block-scaled FP4 GEMM -- test infrastructure.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It wraps ``oracle.c`` (plain C, fp64,
OpenMP over output rows) through ctypes and shares nothing with the CUDA path.

Functions (each follows the passage cited in ``oracle.c``):

* ``e2m1(code)``, ``e4m3(code)``, ``e8m0(code)`` -- exact decoders.
* ``gemm_rows(inp, rows=None)`` -> (D64, absdot) for whole output rows.
* ``gemm_pairs(inp, ii, jj)`` -> (D64, absdot) for sampled output elements.
* ``round_bf16(x)`` -> uint16 bf16 bits (one rounding, ties to even).
* ``scale_reorder(sf, rows, ksf)`` -> the 128x4 atom layout (uint8).
* ``e2m1_encode(q)``, ``e4m3_encode(v)`` -> nearest code (ties to the even code).
* ``epilogue(y, bias, op)`` -> bias, then none / ReLU / squared ReLU / SwiGLU
  (interleaved gate, up columns) on fp64 GEMM results.
* ``quantize(X, fmt)`` -> (packed E2M1 codes, plain row-major scale bytes) of
  fp32 or bf16 values, one scale per 16 (nvfp4) or 32 (mxfp4) values.
* ``grouped_gemm_rows(gin, rows=None)`` -> (D64, absdot): the grouped (MoE)
  GEMM -- independent GEMMs on consecutive row ranges of A and D, group g
  with its own weight matrix B_g.

Parity status of each function is recorded in the module docstrings of
``tests/test_oracle.py``; every function here is pinned there.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_oracle.so")
# The pin-strength test points this at a deliberately mutated copy of the oracle.
_LIB_OVERRIDE = os.environ.get("FP4_ORACLE_LIB")
_lib = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_i64p = ctypes.POINTER(ctypes.c_int64)
_f64p = ctypes.POINTER(ctypes.c_double)
_u16p = ctypes.POINTER(ctypes.c_uint16)


def build(force: bool = False) -> str:
    """Compile oracle.c into _oracle.so next to it (gcc, OpenMP, no FP contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        if _LIB_OVERRIDE:
            lib = ctypes.CDLL(_LIB_OVERRIDE)
        else:
            build()
            lib = ctypes.CDLL(_LIB)
        for name in ("oracle_e2m1", "oracle_e4m3", "oracle_e8m0"):
            f = getattr(lib, name)
            f.argtypes = [ctypes.c_uint]
            f.restype = ctypes.c_double
        lib.oracle_gemm_rows.argtypes = [_u8p, _u8p, _u8p, _u8p, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_int64, ctypes.c_int, ctypes.c_double, _i64p,
                                         ctypes.c_int64, _f64p, _f64p, ctypes.c_int]
        lib.oracle_gemm_rows.restype = ctypes.c_int
        lib.oracle_gemm_pairs.argtypes = [_u8p, _u8p, _u8p, _u8p, ctypes.c_int64, ctypes.c_int64,
                                          ctypes.c_int64, ctypes.c_int, ctypes.c_double, _i64p,
                                          _i64p, ctypes.c_int64, _f64p, _f64p, ctypes.c_int]
        lib.oracle_gemm_pairs.restype = ctypes.c_int
        lib.oracle_round_f32.argtypes = [ctypes.c_double]
        lib.oracle_round_f32.restype = ctypes.c_float
        lib.oracle_round_bf16.argtypes = [ctypes.c_double]
        lib.oracle_round_bf16.restype = ctypes.c_uint16
        lib.oracle_round_bf16_array.argtypes = [_f64p, _u16p, ctypes.c_int64]
        lib.oracle_round_bf16_array.restype = None
        lib.oracle_scale_atom_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
        lib.oracle_scale_atom_bytes.restype = ctypes.c_int64
        lib.oracle_scale_reorder.argtypes = [_u8p, ctypes.c_int64, ctypes.c_int64, _u8p]
        lib.oracle_scale_reorder.restype = None
        lib.oracle_e2m1_encode.argtypes = [ctypes.c_float]
        lib.oracle_e2m1_encode.restype = ctypes.c_uint
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint
        lib.oracle_quantize.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                        ctypes.c_int, _u8p, _u8p]
        lib.oracle_quantize.restype = ctypes.c_int
        lib.oracle_epilogue.argtypes = [_f64p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, _f64p]
        lib.oracle_epilogue.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray, t):
    return a.ctypes.data_as(t)


def e2m1(code: int) -> float:
    return _load().oracle_e2m1(code)


def e4m3(code: int) -> float:
    return _load().oracle_e4m3(code)


def e8m0(code: int) -> float:
    return _load().oracle_e8m0(code)


def _operands(inp):
    A = np.ascontiguousarray(inp.A, dtype=np.uint8)
    sfA = np.ascontiguousarray(inp.sfA, dtype=np.uint8)
    B = np.ascontiguousarray(inp.B, dtype=np.uint8)
    sfB = np.ascontiguousarray(inp.sfB, dtype=np.uint8)
    M, N, K, vec = int(inp.M), int(inp.N), int(inp.K), int(inp.vec)
    assert A.size == M * K // 2 and B.size == N * K // 2
    assert sfA.size == M * (K // vec) and sfB.size == N * (K // vec)
    return A, sfA, B, sfB, M, N, K, vec


def gemm_rows(inp, rows=None, nthreads: int = 0):
    """D (fp64, len(rows) x N, before output rounding) and |alpha|*sum|a b| of the same shape."""
    A, sfA, B, sfB, M, N, K, vec = _operands(inp)
    if rows is None:
        rows_arr = None
        nrows = M
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = rows_arr.size
    D = np.empty((nrows, N), dtype=np.float64)
    absd = np.empty((nrows, N), dtype=np.float64)
    rc = _load().oracle_gemm_rows(_ptr(A, _u8p), _ptr(sfA, _u8p), _ptr(B, _u8p), _ptr(sfB, _u8p),
                                  M, N, K, vec, float(inp.alpha),
                                  None if rows_arr is None else _ptr(rows_arr, _i64p), nrows,
                                  _ptr(D, _f64p), _ptr(absd, _f64p), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gemm_rows rejected its arguments")
    return D, absd


def gemm_pairs(inp, ii, jj, nthreads: int = 0):
    """D[ii[p], jj[p]] (fp64) and |alpha|*sum|a b| for each sampled pair."""
    A, sfA, B, sfB, M, N, K, vec = _operands(inp)
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    assert ii.shape == jj.shape
    out = np.empty(ii.size, dtype=np.float64)
    absd = np.empty(ii.size, dtype=np.float64)
    rc = _load().oracle_gemm_pairs(_ptr(A, _u8p), _ptr(sfA, _u8p), _ptr(B, _u8p), _ptr(sfB, _u8p),
                                   M, N, K, vec, float(inp.alpha), _ptr(ii, _i64p), _ptr(jj, _i64p),
                                   ii.size, _ptr(out, _f64p), _ptr(absd, _f64p), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gemm_pairs rejected its arguments")
    return out, absd


def round_f32(x: float) -> float:
    return float(_load().oracle_round_f32(float(x)))


def round_bf16(x) -> np.ndarray:
    """fp64 values -> bf16 bit patterns (uint16), one rounding to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_round_bf16_array(_ptr(x, _f64p), _ptr(out, _u16p), x.size)
    return out


def scale_atom_bytes(rows: int, ksf: int) -> int:
    return int(_load().oracle_scale_atom_bytes(rows, ksf))


def scale_reorder(sf: np.ndarray, rows: int, ksf: int) -> np.ndarray:
    """Row-major sf[rows][ksf] (uint8) -> the 128x4 atom layout (uint8, zero padded)."""
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    assert sf.size == rows * ksf
    out = np.empty(scale_atom_bytes(rows, ksf), dtype=np.uint8)
    _load().oracle_scale_reorder(_ptr(sf, _u8p), rows, ksf, _ptr(out, _u8p))
    return out


def e2m1_encode(q: float) -> int:
    return int(_load().oracle_e2m1_encode(float(q)))


def e4m3_encode(v: float) -> int:
    return int(_load().oracle_e4m3_encode(float(v)))


def quantize(X: np.ndarray, fmt: str) -> tuple[np.ndarray, np.ndarray]:
    """X: [rows][K] float32 values, or uint16 bf16 bit patterns -> (codes [rows][K/2],
    scales [rows][K/vec]) with vec 16 (nvfp4, E4M3) or 32 (mxfp4, E8M0)."""
    X = np.ascontiguousarray(X)
    assert X.ndim == 2 and X.dtype in (np.float32, np.uint16)
    rows, K = X.shape
    vec = 16 if fmt == "nvfp4" else 32
    codes = np.empty((rows, K // 2), dtype=np.uint8)
    sf = np.empty((rows, K // vec), dtype=np.uint8)
    rc = _load().oracle_quantize(X.ctypes.data, int(X.dtype == np.uint16), rows, K, vec,
                                 _ptr(codes, _u8p), _ptr(sf, _u8p))
    if rc != 0:
        raise ValueError("oracle_quantize rejected its arguments")
    return codes, sf


EPILOGUE_OPS = {"none": 0, "relu": 1, "relu2": 2, "swiglu": 3}


def epilogue(y: np.ndarray, bias, op: str) -> np.ndarray:
    """y: [rows][N] fp64 (alpha already applied); bias: float32 [N] or None.
    Returns [rows][N] (or [rows][N/2] for swiglu) fp64, before output rounding."""
    y = np.ascontiguousarray(y, dtype=np.float64)
    rows, N = y.shape
    code = EPILOGUE_OPS[op]
    out = np.empty((rows, N // 2 if code == 3 else N), dtype=np.float64)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    rc = _load().oracle_epilogue(_ptr(y, _f64p), rows, N, None if b is None else b.ctypes.data, code,
                                 _ptr(out, _f64p))
    if rc != 0:
        raise ValueError("oracle_epilogue rejected its arguments")
    return out


# ---- grouped GEMM (mixture-of-experts layers) --------------------------------
#
# A grouped GEMM is a set of independent GEMMs sharing N and K: group g owns
# rows offsets[g] .. offsets[g+1]-1 of A (and of D) and the weight matrix B_g,
# rows g*N .. g*N+N-1 of the stacked B (the NVFP4 ReLU-squared MoE workload of
# "TMA Pipelines, Tensor Cores, and ctm-rs Interop", "Where to Go Next": each
# expert applies its own weights to the tokens routed to it). Each group's
# rows are computed by gemm_rows on that group's slices -- nothing else.

class _GroupProblem:
    """One group's GEMM as gemm_rows takes it."""

    def __init__(self, gin, g):
        o0, o1 = int(gin.offsets[g]), int(gin.offsets[g + 1])
        K, vec, N = int(gin.K), int(gin.vec), int(gin.N)
        self.A = gin.A.reshape(-1, K // 2)[o0:o1]
        self.sfA = gin.sfA.reshape(-1, K // vec)[o0:o1]
        self.B = gin.B.reshape(-1, K // 2)[g * N:(g + 1) * N]
        self.sfB = gin.sfB.reshape(-1, K // vec)[g * N:(g + 1) * N]
        self.M, self.N, self.K, self.vec, self.alpha = o1 - o0, N, K, vec, gin.alpha


def _group_of_rows(offsets: np.ndarray, rows: np.ndarray) -> np.ndarray:
    """Group of each D row: the g with offsets[g] <= row < offsets[g+1]."""
    return np.searchsorted(offsets, rows, side="right") - 1


def grouped_gemm_rows(gin, rows=None, nthreads: int = 0):
    """D rows (fp64, before output rounding) and |alpha|*sum|a b| of a grouped
    GEMM. gin: fmt, offsets (G+1, int64), N, K, vec, alpha, A [M_total][K/2],
    sfA [M_total][K/vec], B [G*N][K/2], sfB [G*N][K/vec]."""
    offsets = np.asarray(gin.offsets, dtype=np.int64)
    m_total = int(offsets[-1])
    rows = np.arange(m_total, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    D = np.empty((rows.size, int(gin.N)), dtype=np.float64)
    absd = np.empty_like(D)
    groups = _group_of_rows(offsets, rows)
    for g in np.unique(groups):
        sel = np.nonzero(groups == g)[0]
        d, a = gemm_rows(_GroupProblem(gin, int(g)), rows[sel] - offsets[g], nthreads=nthreads)
        D[sel], absd[sel] = d, a
    return D, absd
