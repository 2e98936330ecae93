"""GPU parity at the edges of the index ranges: a long K, and outputs with more
than 2^31 elements (64-bit addressing in every store path).

Same tolerances as tests/test_gemm_gpu.py. The large outputs are checked on
sampled rows gathered on the device (every element of the rows past element
2^31 and of the last row), and a guard region after D must stay untouched.
"""
from __future__ import annotations

import numpy as np
import pytest

import workloads as W
from tests.test_gemm_gpu import check_full, check_sampled, check_values, run

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

GUARD = 4096


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


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_long_k_swap_split(fp4, orc, fmt):
    # K = 2^20 (4096 k-tiles); the skinny plan splits K and reduces
    inp = W.make_random(fmt, 5, 136, 1 << 20, out="f32", alpha=0.25, seed=81)
    check_full(orc, inp, run(fp4, inp), "long K %s" % fmt)


def test_long_k_direct(fp4, orc):
    # K = 2^18 in direct mode, one CTA per MMA with the split last wave
    inp = W.make_random("nvfp4", 384, 768, 1 << 18, out="bf16", seed=82, name="long_k_direct")
    cfg = fp4.GemmConfig(mode=1, bn=256, cta_group=1, max_ctas=6)   # 9 tiles on 6 CTAs: 3 split
    check_sampled(orc, inp, run(fp4, inp, cfg), n_random=4, n_pairs=2000)


def _large_output(fp4, orc, inp, fmt):
    M, N = inp.M, inp.N
    assert M * N > 2 ** 31
    dt = torch.float32 if inp.out == "f32" else torch.bfloat16
    flat = torch.full((M * N + GUARD,), float("nan"), dtype=dt, device="cuda")
    D = flat[:M * N].view(M, N)
    A, sfA, B, sfB = (_dev(getattr(inp, k)) for k in ("A", "sfA", "B", "sfB"))
    fp4.gemm(fmt, A, sfA, B, sfB, inp.alpha, D, M, N, inp.K, inp.out)
    st = fp4.get_device_status()
    assert st == fp4.FP4_OK, fp4.status_string(st)
    first_past = (2 ** 31) // N                      # rows holding elements past index 2^31
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, M // 2], np.arange(first_past, M), rng.integers(0, M, 3)]))
    got = D[torch.from_numpy(rows).cuda()]
    got = got.cpu().numpy().astype(np.float64) if inp.out == "f32" else \
        got.view(torch.int16).cpu().numpy().view(np.uint16)
    ref, absd = orc.gemm_rows(inp, rows)
    check_values(orc, inp.out, got, ref, absd, "rows past 2^31 elements")
    guard = flat[M * N:]
    assert torch.isnan(guard.float()).all(), "written past the end of D"


def test_output_past_2pow31_direct(fp4, orc):
    # 65541 x 32800 bf16 (2.15e9 elements, 4.3 GB): direct-mode row stores
    inp = W.make_random("nvfp4", 65541, 32800, 64, out="bf16", seed=83, name="d_past_2pow31")
    assert fp4.gemm_plan("nvfp4", inp.M, inp.N, inp.K, "bf16")["swap"] is False
    _large_output(fp4, orc, inp, "nvfp4")


def test_output_past_2pow31_swap(fp4, orc):
    # 256 x 8400000 fp32 (2.15e9 elements, 8.6 GB): swap-AB transposed stores
    inp = W.make_random("mxfp4", 256, 8400000, 32, out="f32", seed=84, name="dt_past_2pow31")
    assert fp4.gemm_plan("mxfp4", inp.M, inp.N, inp.K, "f32")["swap"] is True
    _large_output(fp4, orc, inp, "mxfp4")
