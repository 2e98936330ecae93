"""The C-ABI library without a GPU: it builds, loads, exports every symbol that
include/fp4_gemm.h declares, and rejects bad arguments on the host before any
CUDA call. No compute call is made here."""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("fp4_gemm.h", "fp4_quant.h")]


@pytest.fixture(scope="module")
def fp4():
    import block_scaled_fp4_sfa_gb300 as m
    m.build()
    return m


def declared_functions():
    text = "".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp4_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("fp4_gemm_nvfp4", "fp4_gemm_mxfp4", "fp4_gemm_nvfp4_prepacked", "fp4_gemm_mxfp4_prepacked",
                 "fp4_scale_atom_bytes", "fp4_scale_reorder", "fp4_get_device_status", "fp4_status_string",
                 "fp4_quantize"):
        assert must in names


def test_library_exports_every_declared_symbol(fp4):
    lib = fp4.load()
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_library_is_sm103a_only(fp4):
    # the fatbin carries sm_103a SASS; the build flags name exactly one -gencode
    from block_scaled_fp4_sfa_gb300 import _build
    assert _build.ARCH == "-gencode=arch=compute_103a,code=sm_103a"
    assert os.path.getsize(_build.LIB) > 0


def test_status_strings(fp4):
    # every declared status, FP4_OK .. FP4_ERR_SCRATCH_LIMIT, has its own text
    texts = [fp4.status_string(code) for code in range(8)]
    assert all(texts) and len(set(texts)) == 8
    assert "static scratch" in texts[7]
    assert fp4.status_string(99) == "unknown status"


@pytest.mark.parametrize("rows,K,vec", [(1, 32, 16), (128, 256, 16), (129, 288, 16), (300, 96, 32), (0, 64, 16)])
def test_scale_atom_bytes(fp4, rows, K, vec):
    import oracle
    assert fp4.scale_atom_bytes(rows, K, vec) == oracle.scale_atom_bytes(rows, K // vec)


def test_scale_atom_bytes_rejects(fp4):
    assert fp4.scale_atom_bytes(10, 48, 32) == 0
    assert fp4.scale_atom_bytes(10, 64, 8) == 0
    assert fp4.scale_atom_bytes(-1, 64, 16) == 0


def _g(fp4, *args, cfg=None):
    lib = fp4.load()
    fmt, A, sfA, B, sfB, alpha, D, M, N, K, out = args
    return lib.fp4_gemm(fmt, 0, A, sfA, B, sfB, alpha, D, M, N, K, out,
                        ctypes.byref(cfg) if cfg is not None else None, 0)


def test_host_validation_without_device(fp4):
    buf = np.zeros(4096 + 16, np.uint8)
    p = buf.ctypes.data + (-buf.ctypes.data) % 16          # 16-byte aligned address
    # empty problems are no-ops
    assert _g(fp4, 0, p, p, p, p, 1.0, p, 0, 64, 64, 0) == 0
    assert _g(fp4, 0, p, p, p, p, 1.0, p, 64, 0, 64, 0) == 0
    # bad enums, sizes and pointers
    assert _g(fp4, 7, p, p, p, p, 1.0, p, 64, 64, 64, 0) == 1
    assert _g(fp4, 0, p, p, p, p, 1.0, p, 64, 64, 64, 5) == 1
    assert _g(fp4, 0, p, p, p, p, 1.0, p, -1, 64, 64, 0) == 1
    assert _g(fp4, 0, None, p, p, p, 1.0, p, 64, 64, 64, 0) == 1
    assert _g(fp4, 0, p, p, p, p, 1.0, None, 64, 64, 64, 0) == 1
    assert _g(fp4, 0, p, p, p, p, 1.0, p, 64, 64, 48, 0) == 2          # K % 32 != 0
    assert _g(fp4, 0, p + 1, p, p, p, 1.0, p, 64, 64, 64, 0) == 3      # misaligned A
    assert _g(fp4, 0, p, p, p + 8, p, 1.0, p, 64, 64, 64, 0) == 3      # misaligned B
    assert _g(fp4, 0, p, p, p, p, 1.0, p + 4, 64, 64, 64, 0) == 3      # misaligned D
    assert _g(fp4, 0, p, p, p, p, 1.0, p, 1 << 31, 64, 64, 0) == 2     # beyond the index range
    lib = fp4.load()
    assert lib.fp4_scale_reorder(p, p, 10, 48, 32, 0) == 2
    assert lib.fp4_scale_reorder(p, p, -1, 64, 16, 0) == 1
    assert lib.fp4_scale_reorder(p, p + 4, 10, 64, 16, 0) == 3
    assert lib.fp4_scale_reorder(p, p, 0, 64, 16, 0) == 0
    assert lib.fp4_gemm_host(0, p, p, p, p, 1.0, p, 64, 64, 40, 0, 0) == 2
    assert lib.fp4_scale_reorder2(p, p, 10, p, p, 10, 48, 32, 0) == 2
    assert lib.fp4_scale_reorder2(p, p, -1, p, p, 10, 64, 16, 0) == 1
    assert lib.fp4_scale_reorder2(None, p, 10, p, p, 10, 64, 16, 0) == 1
    assert lib.fp4_scale_reorder2(p, p, 10, p, p + 4, 10, 64, 16, 0) == 3
    assert lib.fp4_scale_reorder2(p, p, 0, p, p, 0, 64, 16, 0) == 0


def test_fused_host_validation_without_device(fp4):
    buf = np.zeros(4096 + 16, np.uint8)
    p = buf.ctypes.data + (-buf.ctypes.data) % 16
    lib = fp4.load()

    def f(act, bias, M, N, K=64):
        epi = fp4.Epilogue(act, bias)
        return lib.fp4_gemm_fused(0, 0, p, p, p, p, 1.0, ctypes.byref(epi), p, M, N, K, 0, None, 0)

    assert f(0, None, 0, 64) == 0                  # empty
    assert f(3, None, 64, 0) == 0
    assert f(4, None, 64, 64) == 1                 # unknown activation
    assert f(-1, None, 64, 64) == 1
    assert f(3, None, 64, 63) == 2                 # SwiGLU needs N even
    assert f(1, p + 2, 64, 64) == 3                # bias not 4-byte aligned
    assert f(2, p, 64, 64, K=48) == 2              # K % 32 != 0


def test_plan_host_validation_without_device(fp4):
    lib = fp4.load()
    info = fp4.PlanInfo()

    def plan(fmt=0, M=1, N=64, K=64, out=0, act=0, cfg=None, ptr=True):
        return lib.fp4_gemm_plan(fmt, 0, M, N, K, out, act, cfg, ctypes.byref(info) if ptr else None)

    assert plan(ptr=False) == 1
    assert plan(fmt=3) == 1
    assert plan(out=2) == 1
    assert plan(act=5) == 1
    assert plan(M=-1) == 1
    assert plan(K=40) == 2
    assert plan(N=63, act=3) == 2
    info.launches = 7
    assert plan(M=0) == 0 and info.launches == 0          # nothing to launch
    assert plan(cfg=ctypes.byref(fp4.GemmConfig(mode=4))) in (1, 6)   # bad mode (or no device first)
    assert plan(cfg=ctypes.byref(fp4.GemmConfig(split_tail=2))) in (1, 6)   # split_tail is 0 or 1


def test_grouped_host_validation_without_device(fp4):
    buf = np.zeros(4096 + 16, np.uint8)
    p = buf.ctypes.data + (-buf.ctypes.data) % 16
    lib = fp4.load()

    def grp(offs, N=64, K=64, act=0, bias=None, fmt=0, out=0, cfg=None, D=None):
        o = np.ascontiguousarray(offs, dtype=np.int64)
        epi = fp4.Epilogue(act, bias)
        return lib.fp4_gemm_grouped(fmt, 0, o.size - 1, o.ctypes.data if o.size else None, p, p, p, p, 1.0,
                                    ctypes.byref(epi), p if D is None else D, N, K, out, cfg, 0)

    assert lib.fp4_gemm_grouped(0, 0, 0, None, p, p, p, p, 1.0, None, p, 64, 64, 0, None, 0) == 0   # G = 0
    assert grp([0, 0, 0]) == 0                      # every group empty
    assert grp([0, 4, 9], N=0) == 0
    assert grp([1, 4]) == 1                         # offsets[0] != 0
    assert grp([0, 5, 4]) == 1                      # decreasing
    assert grp([0, 4], fmt=2) == 1
    assert grp([0, 4], act=7) == 1
    assert grp([0, 4], N=63, act=3) == 2            # SwiGLU, odd N
    assert grp([0, 4], bias=p + 2, act=1) == 3      # misaligned bias
    assert grp([0, 4], K=48) == 2
    assert grp([0, 4], D=p + 8) == 3                # misaligned D
    assert grp([0, 4], cfg=ctypes.byref(fp4.GemmConfig(mode=5))) == 1
    assert grp([0, 4], cfg=ctypes.byref(fp4.GemmConfig(splits=2))) == 2
    assert lib.fp4_gemm_grouped(0, 0, 2, None, p, p, p, p, 1.0, None, p, 64, 64, 0, None, 0) == 1   # no offsets
    assert grp(np.arange(258)) == 2                 # more than 256 groups
    many = np.arange(258, dtype=np.int64)
    assert lib.fp4_scale_reorder_grouped(p, p, 257, many.ctypes.data, 64, 16, 0) == 2


def test_quantize_host_validation_without_device(fp4):
    buf = np.zeros(4096 + 16, np.uint8)
    p = buf.ctypes.data + (-buf.ctypes.data) % 16
    q = fp4.load().fp4_quantize
    # no-ops
    assert q(0, p, 1, 0, 64, p, p, 0, 0) == 0
    assert q(0, p, 1, 8, 0, p, p, 1, 0) == 0
    # enums, sizes, pointers, alignment
    assert q(2, p, 1, 8, 64, p, p, 0, 0) == 1
    assert q(0, p, 2, 8, 64, p, p, 0, 0) == 1
    assert q(0, p, 1, 8, 64, p, p, 2, 0) == 1
    assert q(0, p, 1, -1, 64, p, p, 0, 0) == 1
    assert q(0, p, 1, 8, 48, p, p, 0, 0) == 2            # K % 32 != 0
    assert q(0, None, 1, 8, 64, p, p, 0, 0) == 1
    assert q(1, p, 1, 8, 64, p, None, 0, 0) == 1
    assert q(0, p + 2, 1, 8, 64, p, p, 0, 0) == 3        # X not 16-byte aligned
    assert q(0, p, 1, 8, 64, p + 8, p, 0, 0) == 3        # codes not 16-byte aligned
    assert q(0, p, 1, 8, 64, p, p + 4, 1, 0) == 3        # atom scales not 16-byte aligned
    assert q(0, p, 1, 1 << 40, 64, p, p, 0, 0) == 2      # beyond the index range


def test_python_binding_raises(fp4):
    buf = np.zeros(64, np.uint8)
    with pytest.raises(fp4.Fp4Error) as e:
        fp4.gemm("nvfp4", buf, buf, buf, buf, 1.0, buf, 4, 4, 48, "f32", stream=0)
    assert e.value.status == 2


def test_package_fails_loudly_without_library(tmp_path, monkeypatch):
    import block_scaled_fp4_sfa_gb300 as m
    monkeypatch.setattr(m, "_lib", None)
    monkeypatch.setattr(m._build, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        m.load()


def test_grouped_atom_bytes_without_device(fp4):
    import oracle
    offsets = np.array([0, 130, 130, 131, 400], np.int64)
    want = sum(oracle.scale_atom_bytes(int(b - a), 256 // 16) for a, b in zip(offsets[:-1], offsets[1:]) if b > a)
    assert fp4.scale_atom_bytes_grouped(offsets, 256, 16) == want
    assert fp4.scale_atom_bytes_grouped([0, 5, 3], 256, 16) == 0        # decreasing
    assert fp4.scale_atom_bytes_grouped([0, 5], 48, 32) == 0            # K % vec
    assert fp4.scale_atom_bytes_grouped([0], 256, 16) == 0              # no groups
