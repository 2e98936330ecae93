"""fp4_gemm_static_scratch: the GEMM for callers that must not allocate device
memory. Its scratch (reordered scales, split-K partials) is the library's
static 16 MiB device array instead of stream-ordered allocations.

Checked through the C ABI against the allocating entry point on the same
inputs, twice in a row (the second call finds the first call's bytes in the
shared array), with the parity tolerances of the other GPU tests. Named to be
collected last, so a stop-at-first-failure run has done everything else first.
"""
from __future__ import annotations

import numpy as np
import pytest

import workloads as W
from tests._helpers import bf16_bits_to_f64, bf16_ulp

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


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _call(fp4, entry, inp, tensors):
    dt = torch.float32 if inp.out == "f32" else torch.bfloat16
    D = torch.full((inp.M, inp.N), float("nan"), dtype=dt, device="cuda")
    A, sfA, B, sfB = tensors
    if entry == "static":
        fp4.gemm_static_scratch(inp.fmt, A, sfA, B, sfB, inp.alpha, D, inp.M, inp.N, inp.K, inp.out)
    else:
        named = fp4.gemm_nvfp4 if inp.fmt == "nvfp4" else fp4.gemm_mxfp4
        named(A, sfA, B, sfB, inp.alpha, D, inp.M, inp.N, inp.K, inp.out)
    assert fp4.get_device_status() == fp4.FP4_OK
    if inp.out == "f32":
        return D.cpu().numpy().astype(np.float64)
    return D.view(torch.int16).cpu().numpy().view(np.uint16)


def _within_tolerance(inp, got, ref):
    if inp.out == "f32":
        import oracle
        oracle.build()
        _, absd = oracle.gemm_rows(inp)
        assert np.all(np.abs(got - ref) <= 1e-5 * absd + 1e-6)
    else:
        assert np.all(np.abs(bf16_bits_to_f64(got) - bf16_bits_to_f64(ref)) <= bf16_ulp(ref))


# direct plan with reordered scales; swap-AB plan with split-K partials
CASES = [("nvfp4", 300, 520, 1024, "f32"), ("mxfp4", 16, 1536, 2048, "bf16"), ("nvfp4", 1, 1000, 4096, "f32")]


@pytest.mark.parametrize("fmt,M,N,K,out", CASES)
def test_static_scratch_matches_allocating_entry(fp4, fmt, M, N, K, out):
    inp = W.make_random(fmt, M, N, K, out=out, seed=M + K)
    tensors = [_dev(getattr(inp, k)) for k in ("A", "sfA", "B", "sfB")]
    ref = _call(fp4, "alloc", inp, tensors)
    for _ in range(2):                                   # two calls in a row share the array
        got = _call(fp4, "static", inp, tensors)
        _within_tolerance(inp, got, ref)


def test_static_scratch_rejects_oversized(fp4):
    # MXFP4 always reorders its scales: at 8192 x 8192 x 65536 the two atom copies
    # take 2 x 64 row blocks x 512 atoms x 512 B = 32 MiB, over the 16 MiB array.
    # Every buffer is real and sized for the problem (all zeros), so the call is
    # a valid GEMM even if it were not refused.
    M = N = 8192
    K = 1 << 16
    A = torch.zeros(M, K // 2, dtype=torch.uint8, device="cuda")
    B = torch.zeros(N, K // 2, dtype=torch.uint8, device="cuda")
    sfA = torch.zeros(M, K // 32, dtype=torch.uint8, device="cuda")
    sfB = torch.zeros(N, K // 32, dtype=torch.uint8, device="cuda")
    D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    st = fp4.gemm_static_scratch("mxfp4", A, sfA, B, sfB, 1.0, D, M, N, K, "bf16", check=False)
    assert st == 7 and "static scratch" in fp4.status_string(st)
    assert fp4.get_device_status() == fp4.FP4_OK
