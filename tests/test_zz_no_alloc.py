"""fp4_gemm_static_scratch: the GEMM for callers that must not allocate device
memory. Its scratch (reordered scales, split-K partials) is the library's
static 16 MiB device array instead of stream-ordered allocations.

Every result is checked through the C ABI twice over: element by element
against the CPU oracle with the parity tolerances of tests/test_gemm_gpu.py
(fp32 output: |D - ref| <= 1e-5 |alpha| sum|a b| + 1e-6; bf16 output: within
1 bf16 ulp of the rounded oracle value), and against the allocating entry point
on the same inputs within the same bounds. Each case runs two calls in a row
(the second finds the first call's bytes in the shared array). Also covered: a
shape whose automatic plan splits K more ways than the array holds (the call
then takes fewer splits instead of refusing), a call recorded into a CUDA graph
and replayed between plain calls, and the refusal of a problem whose scale atoms
alone exceed the array. Named to be collected last, so a stop-at-first-failure
run has done everything else first.
"""
from __future__ import annotations

import numpy as np
import pytest

import workloads as W
from tests._helpers import bf16_bits_to_f64, bf16_ulp
from tests.test_gemm_gpu import check_values

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


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _host(D, out):
    if out == "f32":
        return D.cpu().numpy().astype(np.float64)
    return D.view(torch.int16).cpu().numpy().view(np.uint16)


def _call(fp4, entry, inp, tensors, D=None):
    dt = torch.float32 if inp.out == "f32" else torch.bfloat16
    if D is None:
        D = torch.full((inp.M, inp.N), float("nan"), dtype=dt, device="cuda")
    A, sfA, B, sfB = tensors
    if entry == "static":
        fp4.gemm_static_scratch(inp.fmt, A, sfA, B, sfB, inp.alpha, D, inp.M, inp.N, inp.K, inp.out)
    else:
        named = fp4.gemm_nvfp4 if inp.fmt == "nvfp4" else fp4.gemm_mxfp4
        named(A, sfA, B, sfB, inp.alpha, D, inp.M, inp.N, inp.K, inp.out)
    assert fp4.get_device_status() == fp4.FP4_OK
    return _host(D, inp.out)


def _rows(M):
    return np.unique(np.array([0, 1, M // 3, M // 2, M - 2, M - 1]).clip(0, M - 1))


def _check(orc, inp, got, alloc, rows=None):
    """got against the oracle (all rows, or the given ones) and against the allocating entry."""
    ref, absd = orc.gemm_rows(inp) if rows is None else orc.gemm_rows(inp, rows)
    sel = slice(None) if rows is None else rows
    check_values(orc, inp.out, got[sel], ref, absd, "static scratch vs oracle")
    if inp.out == "f32":
        assert np.all(np.abs(got[sel] - alloc[sel]) <= 1e-5 * absd + 1e-6)
    else:
        assert np.all(np.abs(bf16_bits_to_f64(got[sel]) - bf16_bits_to_f64(alloc[sel])) <= bf16_ulp(alloc[sel]))


# direct plan with reordered scales; swap-AB with split-K partials; the narrow-M
# kernel (no scratch at all)
CASES = [("nvfp4", 300, 520, 1024, "f32"), ("mxfp4", 16, 1536, 2048, "bf16"), ("nvfp4", 1, 1000, 4096, "f32"),
         ("mxfp4", 640, 768, 2048, "bf16")]


@pytest.mark.parametrize("fmt,M,N,K,out", CASES)
def test_static_scratch_matches_oracle_and_allocating_entry(fp4, orc, fmt, M, N, K, out):
    inp = W.make_random(fmt, M, N, K, out=out, seed=M + K)
    tensors = [_dev(getattr(inp, k)) for k in ("A", "sfA", "B", "sfB")]
    alloc = _call(fp4, "alloc", inp, tensors)
    for _ in range(2):                                   # two calls in a row share the array
        got = _call(fp4, "static", inp, tensors)
        _check(orc, inp, got, alloc)


def test_static_scratch_takes_fewer_splits_when_partials_do_not_fit(fp4, orc):
    # 128 x 4096 x 32768 NVFP4: the automatic swap-AB plan splits K (4 ways) so
    # that its fp32 partials (splits x 2 MiB) plus the scale atoms (8.3 MiB)
    # exceed the 16 MiB array; the call must lower the split count, not refuse.
    M, N, K = 128, 4096, 32768
    inp = W.make_random("nvfp4", M, N, K, out="bf16", seed=5)
    plan = fp4.gemm_plan("nvfp4", M, N, K, "bf16")
    atoms = fp4.scale_atom_bytes(M, K, 16) + fp4.scale_atom_bytes(N, K, 16)
    assert plan["swap"] and plan["splits"] > 1
    assert plan["splits"] * M * N * 4 + atoms > fp4.STATIC_SCRATCH_BYTES >= atoms + M * N * 4
    tensors = [_dev(getattr(inp, k)) for k in ("A", "sfA", "B", "sfB")]
    alloc = _call(fp4, "alloc", inp, tensors)
    rows = _rows(inp.M)
    for _ in range(2):
        got = _call(fp4, "static", inp, tensors)
        _check(orc, inp, got, alloc, rows)


def test_static_scratch_replayed_from_a_graph(fp4, orc):
    # The captured call's reordered scales sit in the shared array, which the plain
    # calls between the replays overwrite; every replay must match.
    inp = W.make_random("nvfp4", 300, 520, 1024, out="f32", seed=21)
    tensors = [_dev(getattr(inp, k)) for k in ("A", "sfA", "B", "sfB")]
    alloc = _call(fp4, "alloc", inp, tensors)
    D = torch.full((inp.M, inp.N), float("nan"), dtype=torch.float32, device="cuda")
    _call(fp4, "static", inp, tensors, D)                # first call on the device: set-up, not captured
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    A, sfA, B, sfB = tensors
    with torch.cuda.graph(g, stream=s):
        fp4.gemm_static_scratch(inp.fmt, A, sfA, B, sfB, inp.alpha, D, inp.M, inp.N, inp.K, inp.out)
    torch.cuda.synchronize()
    for _ in range(3):
        D.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert fp4.get_device_status() == fp4.FP4_OK
        _check(orc, inp, _host(D, inp.out), alloc)
        _check(orc, inp, _call(fp4, "static", inp, tensors), alloc)     # a plain call in between


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
