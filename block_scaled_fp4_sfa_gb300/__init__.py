"""Python binding of the GB300 block-scaled FP4 GEMM library (libfp4gemm.so).

Argument marshalling only: every step of the GEMM and of the quantisation that
feeds it runs in the library's CUDA kernels, behind the C ABI declared in
include/fp4_gemm.h and include/fp4_quant.h. Buffers may be torch
tensors (device pointers taken with ``data_ptr()``), numpy arrays (host
pointers, for ``gemm_host``) or raw integer addresses. ``stream`` is a
``torch.cuda.Stream``, a raw ``cudaStream_t`` integer, or None for torch's
current stream.

There is no fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

__all__ = ["FP4_OK", "Fp4Error", "load", "build", "gemm", "gemm_nvfp4", "gemm_mxfp4", "gemm_nvfp4_prepacked",
           "gemm_mxfp4_prepacked", "gemm_host", "scale_reorder", "scale_atom_bytes", "get_device_status",
           "status_string", "set_wait_limit_ms", "GemmConfig", "FMT", "OUT", "gemm_static_scratch",
           "STATIC_SCRATCH_BYTES", "quantize", "IN", "SF_LAYOUT", "gemm_fused", "ACT", "Epilogue", "gemm_plan", "PlanInfo", "gemm_grouped", "scale_reorder_grouped",
           "scale_atom_bytes_grouped", "scale_reorder2"]

FP4_OK = 0
STATUS_NAMES = {0: "FP4_OK", 1: "FP4_ERR_INVALID_ARG", 2: "FP4_ERR_UNSUPPORTED", 3: "FP4_ERR_MISALIGNED",
                4: "FP4_ERR_CUDA", 5: "FP4_ERR_TIMEOUT", 6: "FP4_ERR_NO_DEVICE", 7: "FP4_ERR_SCRATCH_LIMIT"}
STATIC_SCRATCH_BYTES = 16 << 20
FMT = {"nvfp4": 0, "mxfp4": 1}
OUT = {"f32": 0, "bf16": 1}
IN = {"f32": 0, "bf16": 1}
SF_LAYOUT = {"plain": 0, "atom": 1}
ACT = {"none": 0, "relu": 1, "relu2": 2, "swiglu": 3}

_lib = None


class Fp4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s: %s (%s)" % (what, STATUS_NAMES.get(status, status), status_string(status)))


class GemmConfig(ctypes.Structure):
    """fp4_gemm_config: plan overrides (0 = automatic)."""
    _fields_ = [("mode", ctypes.c_int32), ("bn", ctypes.c_int32), ("splits", ctypes.c_int32),
                ("max_ctas", ctypes.c_int32), ("cta_group", ctypes.c_int32), ("stop_after", ctypes.c_int32),
                ("split_tail", ctypes.c_int32)]


class Epilogue(ctypes.Structure):
    """fp4_epilogue: activation code and an optional device bias pointer."""
    _fields_ = [("act", ctypes.c_int32), ("bias", ctypes.c_void_p)]


class PlanInfo(ctypes.Structure):
    """fp4_plan_info: what a call would launch."""
    _fields_ = [("kernel", ctypes.c_int32), ("swap", ctypes.c_int32), ("bn", ctypes.c_int32),
                ("cta_group", ctypes.c_int32), ("splits", ctypes.c_int32), ("launches", ctypes.c_int32)]


def build(force: bool = False) -> str:
    return _build.build(force=force)


def load():
    """Load libfp4gemm.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        raise ImportError("libfp4gemm.so is not built: run __graft_entry__.build() "
                          "(or python block_scaled_fp4_sfa_gb300/_build.py)")
    lib = ctypes.CDLL(_build.LIB)
    vp, i64, f32, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
    gemm_args = [vp, vp, vp, vp, f32, vp, i64, i64, i64, i32, vp]
    for name in ("fp4_gemm_nvfp4", "fp4_gemm_mxfp4", "fp4_gemm_nvfp4_prepacked", "fp4_gemm_mxfp4_prepacked"):
        getattr(lib, name).argtypes = gemm_args
        getattr(lib, name).restype = i32
    lib.fp4_gemm.argtypes = [i32, i32, vp, vp, vp, vp, f32, vp, i64, i64, i64, i32,
                             ctypes.POINTER(GemmConfig), vp]
    lib.fp4_gemm.restype = i32
    lib.fp4_gemm_fused.argtypes = [i32, i32, vp, vp, vp, vp, f32, ctypes.POINTER(Epilogue), vp, i64, i64, i64, i32,
                                   ctypes.POINTER(GemmConfig), vp]
    lib.fp4_gemm_fused.restype = i32
    lib.fp4_gemm_grouped.argtypes = [i32, i32, i64, vp, vp, vp, vp, vp, f32, ctypes.POINTER(Epilogue), vp, i64, i64,
                                     i32, ctypes.POINTER(GemmConfig), vp]
    lib.fp4_gemm_grouped.restype = i32
    lib.fp4_scale_atom_bytes_grouped.argtypes = [i64, vp, i64, i32]
    lib.fp4_scale_atom_bytes_grouped.restype = ctypes.c_size_t
    lib.fp4_scale_reorder_grouped.argtypes = [vp, vp, i64, vp, i64, i32, vp]
    lib.fp4_scale_reorder_grouped.restype = i32
    lib.fp4_gemm_plan.argtypes = [i32, i32, i64, i64, i64, i32, i32, ctypes.POINTER(GemmConfig),
                                  ctypes.POINTER(PlanInfo)]
    lib.fp4_gemm_plan.restype = i32
    lib.fp4_gemm_host.argtypes = [i32, vp, vp, vp, vp, f32, vp, i64, i64, i64, i32, vp]
    lib.fp4_gemm_host.restype = i32
    lib.fp4_gemm_static_scratch.argtypes = [i32, vp, vp, vp, vp, f32, vp, i64, i64, i64, i32, vp]
    lib.fp4_gemm_static_scratch.restype = i32
    lib.fp4_scale_atom_bytes.argtypes = [i64, i64, i32]
    lib.fp4_scale_atom_bytes.restype = ctypes.c_size_t
    lib.fp4_scale_reorder.argtypes = [vp, vp, i64, i64, i32, vp]
    lib.fp4_scale_reorder.restype = i32
    lib.fp4_scale_reorder2.argtypes = [vp, vp, i64, vp, vp, i64, i64, i32, vp]
    lib.fp4_scale_reorder2.restype = i32
    lib.fp4_get_device_status.argtypes = [vp]
    lib.fp4_get_device_status.restype = i32
    lib.fp4_status_string.argtypes = [i32]
    lib.fp4_status_string.restype = ctypes.c_char_p
    lib.fp4_set_wait_limit_ms.argtypes = [i64]
    lib.fp4_set_wait_limit_ms.restype = None
    lib.fp4_quantize.argtypes = [i32, vp, i32, i64, i64, vp, vp, i32, vp]
    lib.fp4_quantize.restype = i32
    _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError("expected a tensor, an array or an address, got %r" % type(x))


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(st: int, what: str):
    if st != FP4_OK:
        raise Fp4Error(st, what)


def status_string(st: int) -> str:
    return load().fp4_status_string(st).decode()


def gemm(fmt: str, A, sfA, B, sfB, alpha: float, D, M: int, N: int, K: int, out: str = "f32", *,
         prepacked: bool = False, config: GemmConfig | None = None, stream=None, check: bool = True) -> int:
    """fp4_gemm: D = alpha * decode(A, sfA) . decode(B, sfB)^T on the device."""
    cfg = ctypes.byref(config) if config is not None else None
    st = load().fp4_gemm(FMT[fmt], int(bool(prepacked)), _ptr(A), _ptr(sfA), _ptr(B), _ptr(sfB), float(alpha),
                         _ptr(D), int(M), int(N), int(K), OUT[out], cfg, _stream(stream))
    if check:
        _check(st, "fp4_gemm")
    return st


def gemm_fused(fmt: str, A, sfA, B, sfB, alpha: float, D, M: int, N: int, K: int, out: str = "f32", *,
               act: str = "none", bias=None, prepacked: bool = False, config: GemmConfig | None = None,
               stream=None, check: bool = True) -> int:
    """fp4_gemm_fused: D = act(alpha * decode(A, sfA) . decode(B, sfB)^T + bias). D has N / 2 columns
    for act="swiglu" (gate and up columns interleaved in B)."""
    epi = Epilogue(ACT[act], _ptr(bias))
    cfg = ctypes.byref(config) if config is not None else None
    st = load().fp4_gemm_fused(FMT[fmt], int(bool(prepacked)), _ptr(A), _ptr(sfA), _ptr(B), _ptr(sfB), float(alpha),
                               ctypes.byref(epi), _ptr(D), int(M), int(N), int(K), OUT[out], cfg, _stream(stream))
    if check:
        _check(st, "fp4_gemm_fused")
    return st


def _offsets(offsets):
    import numpy as np
    return np.ascontiguousarray(np.asarray(offsets, dtype=np.int64))


def scale_reorder2(sf_a, atoms_a, rows_a: int, sf_b, atoms_b, rows_b: int, K: int, vec: int, stream=None,
                   check: bool = True) -> int:
    """fp4_scale_reorder2: both operands' scales in one launch."""
    st = load().fp4_scale_reorder2(_ptr(sf_a), _ptr(atoms_a), int(rows_a), _ptr(sf_b), _ptr(atoms_b), int(rows_b),
                                   int(K), int(vec), _stream(stream))
    if check:
        _check(st, "fp4_scale_reorder2")
    return st


def scale_atom_bytes_grouped(offsets, K: int, vec: int) -> int:
    offs = _offsets(offsets)
    return int(load().fp4_scale_atom_bytes_grouped(int(offs.size - 1), offs.ctypes.data, int(K), int(vec)))


def scale_reorder_grouped(sf, out, offsets, K: int, vec: int, stream=None, check: bool = True) -> int:
    """fp4_scale_reorder_grouped: activation scales -> the grouped atom layout."""
    offs = _offsets(offsets)
    st = load().fp4_scale_reorder_grouped(_ptr(sf), _ptr(out), int(offs.size - 1), offs.ctypes.data, int(K),
                                          int(vec), _stream(stream))
    if check:
        _check(st, "fp4_scale_reorder_grouped")
    return st


def gemm_grouped(fmt: str, offsets, A, sfA, B, sfB, alpha: float, D, N: int, K: int, out: str = "f32", *,
                 act: str = "none", bias=None, weights_prepacked: bool = False, acts_prepacked: bool = False,
                 config: GemmConfig | None = None, stream=None, check: bool = True) -> int:
    """fp4_gemm_grouped: group g = rows offsets[g] .. offsets[g+1]-1 of A and D, weights B[g]. ``offsets``
    is a host sequence of G + 1 integers; bias, if given, is [G][N] on the device."""
    offs = _offsets(offsets)
    epi = Epilogue(ACT[act], _ptr(bias))
    cfg = ctypes.byref(config) if config is not None else None
    flags = (1 if weights_prepacked else 0) | (2 if acts_prepacked else 0)
    st = load().fp4_gemm_grouped(FMT[fmt], flags, int(offs.size - 1), offs.ctypes.data,
                                 _ptr(A), _ptr(sfA), _ptr(B), _ptr(sfB), float(alpha), ctypes.byref(epi), _ptr(D),
                                 int(N), int(K), OUT[out], cfg, _stream(stream))
    if check:
        _check(st, "fp4_gemm_grouped")
    return st


def gemm_plan(fmt: str, M: int, N: int, K: int, out: str = "f32", *, act: str = "none", prepacked: bool = False,
              config: GemmConfig | None = None) -> dict:
    """fp4_gemm_plan: {"kernel": "tcgen05" | "narrow", "swap", "bn", "cta_group", "splits", "launches"}."""
    info = PlanInfo()
    cfg = ctypes.byref(config) if config is not None else None
    _check(load().fp4_gemm_plan(FMT[fmt], int(bool(prepacked)), int(M), int(N), int(K), OUT[out], ACT[act], cfg,
                                ctypes.byref(info)), "fp4_gemm_plan")
    return {"kernel": "narrow" if info.kernel == 1 else "tcgen05", "swap": bool(info.swap), "bn": info.bn,
            "cta_group": info.cta_group, "splits": info.splits, "launches": info.launches}


def _named(name):
    def call(A, sfA, B, sfB, alpha, D, M, N, K, out="f32", stream=None, check=True):
        st = getattr(load(), name)(_ptr(A), _ptr(sfA), _ptr(B), _ptr(sfB), float(alpha), _ptr(D), int(M), int(N),
                                   int(K), OUT[out], _stream(stream))
        if check:
            _check(st, name)
        return st
    call.__name__ = name
    return call


gemm_nvfp4 = _named("fp4_gemm_nvfp4")
gemm_mxfp4 = _named("fp4_gemm_mxfp4")
gemm_nvfp4_prepacked = _named("fp4_gemm_nvfp4_prepacked")
gemm_mxfp4_prepacked = _named("fp4_gemm_mxfp4_prepacked")


def gemm_host(fmt: str, A, sfA, B, sfB, alpha: float, D, M: int, N: int, K: int, out: str = "f32",
              stream=None, check: bool = True) -> int:
    """fp4_gemm_host: host buffers in and out (pinned memory for asynchronous copies)."""
    st = load().fp4_gemm_host(FMT[fmt], _ptr(A), _ptr(sfA), _ptr(B), _ptr(sfB), float(alpha), _ptr(D), int(M),
                              int(N), int(K), OUT[out], _stream(stream))
    if check:
        _check(st, "fp4_gemm_host")
    return st


def gemm_static_scratch(fmt: str, A, sfA, B, sfB, alpha: float, D, M: int, N: int, K: int, out: str = "f32",
                        stream=None, check: bool = True) -> int:
    """fp4_gemm_static_scratch: plain-scale GEMM for callers that must not allocate;
    its scratch is the library's static 16 MiB device array (see the header)."""
    st = load().fp4_gemm_static_scratch(FMT[fmt], _ptr(A), _ptr(sfA), _ptr(B), _ptr(sfB), float(alpha), _ptr(D),
                                        int(M), int(N), int(K), OUT[out], _stream(stream))
    if check:
        _check(st, "fp4_gemm_static_scratch")
    return st


def scale_atom_bytes(rows: int, k: int, vec: int) -> int:
    return int(load().fp4_scale_atom_bytes(int(rows), int(k), int(vec)))


def scale_reorder(sf, sf_atom, rows: int, k: int, vec: int, stream=None, check: bool = True) -> int:
    st = load().fp4_scale_reorder(_ptr(sf), _ptr(sf_atom), int(rows), int(k), int(vec), _stream(stream))
    if check:
        _check(st, "fp4_scale_reorder")
    return st


def quantize(fmt: str, X, rows: int, K: int, codes, sf, *, in_dtype: str = "bf16", layout: str = "plain",
             stream=None, check: bool = True) -> int:
    """fp4_quantize: X [rows][K] (fp32 or bf16) -> E2M1 codes [rows][K/2] and scale bytes
    (plain [rows][K/vec], or the 128x4 atom layout for the prepacked GEMM calls)."""
    st = load().fp4_quantize(FMT[fmt], _ptr(X), IN[in_dtype], int(rows), int(K), _ptr(codes), _ptr(sf),
                             SF_LAYOUT[layout], _stream(stream))
    if check:
        _check(st, "fp4_quantize")
    return st


def get_device_status(stream=None) -> int:
    return int(load().fp4_get_device_status(_stream(stream)))


def set_wait_limit_ms(ms: int) -> None:
    load().fp4_set_wait_limit_ms(int(ms))
