"""GPU parity of the narrow-M (M <= 4) CUDA-core kernel against the CPU oracle.

Same tolerances as the tcgen05 GEMM (tests/test_gemm_gpu.py): fp32 output
|D - ref| <= 1e-5 * |alpha| * sum_k |a_k b_k| + 1e-6; bf16 output within one
bf16 ulp of the once-rounded oracle value; fused epilogues as in
tests/test_fused_gpu.py. Covered: M = 1..4, both formats, plain and atom-layout
scales, K not a multiple of the kernel's 1024-code pass, odd N, extreme scale
bytes, the fused epilogues, the planner's choice, and agreement with the
tcgen05 path on the same problem.
"""
from __future__ import annotations

import numpy as np
import pytest

import workloads as W
from tests.test_fused_gpu import check as check_fused, expected as expected_fused, run_fused
from tests.test_gemm_gpu import check_full, run

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def fp4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_scaled_fp4_sfa_gb300 as m
    m.build()
    m.load()
    return m


@pytest.fixture(scope="module")
def orc():
    import oracle
    oracle.build()
    return oracle


def narrow(fp4):
    return fp4.GemmConfig(mode=3)


# fmt, out, M, N, K
SHAPES = [
    ("nvfp4", "f32", 1, 1, 32),            # smallest: one block, one lane active
    ("nvfp4", "f32", 1, 300, 4096),        # one full chunk
    ("nvfp4", "bf16", 2, 257, 1056),       # a partial chunk; odd N
    ("nvfp4", "f32", 3, 130, 3104),        # three rows, ragged chunk
    ("nvfp4", "bf16", 4, 64, 8192),        # two 4096-code chunks
    ("nvfp4", "f32", 1, 77, 4128),         # a chunk plus one piece
    ("mxfp4", "f32", 1, 511, 4096),
    ("mxfp4", "bf16", 2, 96, 96),
    ("mxfp4", "f32", 3, 33, 5120),
    ("mxfp4", "f32", 4, 200, 2080),
]


@pytest.mark.parametrize("prepacked", [False, True], ids=["plain", "atoms"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "%s_%s_%dx%dx%d" % s)
def test_narrow_parity(fp4, orc, shape, prepacked):
    fmt, out, M, N, K = shape
    inp = W.make_random(fmt, M, N, K, out=out, alpha=0.5, dist="t3", seed=M * 7 + N + K)
    assert fp4.gemm_plan(fmt, M, N, K, out)["kernel"] == ("narrow" if M == 1 else "tcgen05")
    got = run(fp4, inp, narrow(fp4), prepacked=prepacked)
    check_full(orc, inp, got, "narrow %s" % (shape,))


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_narrow_every_code_and_scale(fp4, orc, fmt):
    # every E2M1 code on both sides; scales 2^u over the normal E4M3 range, or
    # over 2^+-50 for E8M0 (wider would overflow the fp32 result), then E4M3
    # subnormals and zeros (NVFP4) or the byte 0 = 2^-127 (MXFP4) planted in
    # B's scales
    inp = W.make_uniform_codes(fmt, 4, 777, 2048, seed=5, u_range=(-6, 8) if fmt == "nvfp4" else (-50, 50))
    check_full(orc, inp, run(fp4, inp, narrow(fp4)), "codes %s" % fmt)
    inp = W.make_uniform_codes(fmt, 1, 64, 1024, seed=6, u_range=(-3, 3))
    sf = inp.sfB.copy()
    rng = np.random.default_rng(7)
    pick = rng.random(sf.shape) < 0.3
    sf[pick] = rng.integers(0, 8, int(pick.sum())) if fmt == "nvfp4" else 0
    inp.sfB = sf
    check_full(orc, inp, run(fp4, inp, narrow(fp4)), "small scales %s" % fmt)


@pytest.mark.parametrize("act", ["none", "relu", "relu2", "swiglu"])
@pytest.mark.parametrize("with_bias", [False, True], ids=["nobias", "bias"])
@pytest.mark.parametrize("M", [1, 3])
def test_narrow_fused(fp4, orc, M, with_bias, act):
    N, K = 1000, 2048
    inp = W.make_random("nvfp4", M, N, K, out="f32", alpha=0.75, b_std=0.3, seed=M + 40)
    bias = W.make_bias(N, std=1.0, seed=3) if with_bias else None
    got = run_fused(fp4, inp, act, bias, narrow(fp4))
    y, absd = orc.gemm_rows(inp)
    ref, tol = expected_fused(orc, y, absd, bias, act)
    check_fused(orc, inp.out, got, ref, tol, "narrow fused M=%d %s" % (M, act))


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_narrow_matches_tensor_path(fp4, orc, fmt):
    # the same problem through both kernels: each within tolerance of the oracle
    inp = W.make_random(fmt, 2, 1536, 4096, out="f32", seed=9)
    a = run(fp4, inp, narrow(fp4))
    b = run(fp4, inp, fp4.GemmConfig(mode=2))
    check_full(orc, inp, a, "narrow")
    check_full(orc, inp, b, "tcgen05")
    assert np.max(np.abs(a - b)) <= 1e-4 * np.max(np.abs(b))


def test_narrow_deterministic(fp4):
    inp = W.make_random("nvfp4", 1, 28672, 4096, out="f32", dist="t3", seed=2)
    np.testing.assert_array_equal(run(fp4, inp, None), run(fp4, inp, None))


def test_plan_choice(fp4):
    assert fp4.gemm_plan("nvfp4", 1, 28672, 4096)["kernel"] == "narrow"
    assert fp4.gemm_plan("nvfp4", 1, 28672, 4096)["launches"] == 1
    assert fp4.gemm_plan("mxfp4", 1, 100, 8192, "bf16")["kernel"] == "narrow"
    assert fp4.gemm_plan("mxfp4", 2, 100, 8192, "bf16")["kernel"] == "tcgen05"
    assert fp4.gemm_plan("nvfp4", 1, 100, 4096, prepacked=True)["kernel"] == "tcgen05"
    assert fp4.gemm_plan("nvfp4", 3, 100, 4096)["kernel"] == "tcgen05"
    assert fp4.gemm_plan("nvfp4", 4, 100, 4096, config=fp4.GemmConfig(mode=3))["kernel"] == "narrow"
    assert fp4.gemm_plan("nvfp4", 1, 100, 4096, config=fp4.GemmConfig(mode=2))["kernel"] == "tcgen05"
    p = fp4.gemm_plan("nvfp4", 4096, 4096, 4096, "bf16")
    assert p["kernel"] == "tcgen05" and not p["swap"] and p["launches"] == 2     # reorder + GEMM
    assert fp4.gemm_plan("nvfp4", 4096, 4096, 4096, "bf16", prepacked=True)["launches"] == 1
    with pytest.raises(fp4.Fp4Error):
        fp4.gemm_plan("nvfp4", 5, 100, 4096, config=fp4.GemmConfig(mode=3))     # M > 4
    with pytest.raises(fp4.Fp4Error):
        fp4.gemm_plan("nvfp4", 1, 100, 1 << 20, config=fp4.GemmConfig(mode=3))  # A does not fit
    # too long for the staging: the tcgen05 path takes it
    assert fp4.gemm_plan("nvfp4", 1, 100, 1 << 20)["kernel"] == "tcgen05"


def test_narrow_odd_scale_address(fp4, orc):
    # B's scales at an odd address: the narrow kernel reads scale pairs as 16-bit
    # words, so the automatic plan falls back to the tcgen05 path; forcing it fails
    inp = W.make_random("nvfp4", 1, 96, 4128, out="f32", seed=12)
    A, sfA, B = (torch.from_numpy(np.ascontiguousarray(getattr(inp, k))).cuda() for k in ("A", "sfA", "B"))
    buf = torch.zeros(inp.sfB.size + 1, dtype=torch.uint8, device="cuda")
    buf[1:] = torch.from_numpy(inp.sfB.reshape(-1)).cuda()
    odd = buf.data_ptr() + 1
    D = torch.full((1, 96), float("nan"), device="cuda")
    fp4.gemm("nvfp4", A, sfA, B, odd, inp.alpha, D, 1, 96, inp.K, "f32")
    assert fp4.get_device_status() == fp4.FP4_OK
    check_full(orc, inp, D.cpu().numpy().astype(np.float64), "odd sfB")
    with pytest.raises(fp4.Fp4Error) as e:
        fp4.gemm("nvfp4", A, sfA, B, odd, inp.alpha, D, 1, 96, inp.K, "f32", config=narrow(fp4))
    assert e.value.status == 3
