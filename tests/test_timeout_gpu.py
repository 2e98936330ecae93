"""Failure detection on the GPU without a fault: a bounded wait that runs out.

The test-only config field `stop_after` makes every TMA producer of the GEMM
kernel stop after filling that many k-tile stages, so nothing ever lands in the
next stage and the MMA issuer's bounded wait for it runs out (the wait limit is
lowered to a few milliseconds first). No MMA reads a stage that did not land,
nothing faults or traps: the launch records FP4_ERR_TIMEOUT in the device status
word, every role leaves its loop, the kernel waits for the copies and MMAs it did
issue, frees its TMEM and returns. The test checks the status (and that reading
it clears it), then that a normal call on the same stream still matches the CPU
oracle element by element (tolerances as tests/test_gemm_gpu.py).
"""
from __future__ import annotations

import numpy as np
import pytest

import workloads as W
from tests.test_gemm_gpu import check_full

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

FP4_ERR_TIMEOUT = 5


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


# (fmt, M, N, K, out, mode, bn, cta_group, splits): one CTA per MMA, a CTA pair,
# swap-AB with split-K partials
CASES = [("nvfp4", 256, 512, 2048, "f32", 1, 256, 1, 0),
         ("mxfp4", 512, 512, 2048, "bf16", 1, 256, 2, 0),
         ("nvfp4", 64, 1024, 4096, "f32", 2, 64, 1, 2)]


@pytest.mark.parametrize("fmt,M,N,K,out,mode,bn,cg,splits", CASES)
def test_bounded_wait_runs_out_then_recovers(fp4, orc, fmt, M, N, K, out, mode, bn, cg, splits):
    inp = W.make_random(fmt, M, N, K, out=out, seed=M + N)
    A, sfA, B, sfB = (_dev(getattr(inp, k)) for k in ("A", "sfA", "B", "sfB"))
    dt = torch.float32 if out == "f32" else torch.bfloat16
    D = torch.zeros(M, N, dtype=dt, device="cuda")
    assert fp4.get_device_status() == fp4.FP4_OK          # nothing pending from earlier tests
    fp4.set_wait_limit_ms(5)
    try:
        cfg = fp4.GemmConfig(mode=mode, bn=bn, cta_group=cg, splits=splits, stop_after=2)
        fp4.gemm(fmt, A, sfA, B, sfB, inp.alpha, D, M, N, K, out, config=cfg)
        assert fp4.get_device_status() == FP4_ERR_TIMEOUT
        assert fp4.get_device_status() == fp4.FP4_OK      # reading the status cleared it
    finally:
        fp4.set_wait_limit_ms(2000)
    # the context and the library still work: the same call without the stop
    D.fill_(float("nan"))
    cfg = fp4.GemmConfig(mode=mode, bn=bn, cta_group=cg, splits=splits)
    fp4.gemm(fmt, A, sfA, B, sfB, inp.alpha, D, M, N, K, out, config=cfg)
    assert fp4.get_device_status() == fp4.FP4_OK
    got = D.cpu().numpy().astype(np.float64) if out == "f32" else D.view(torch.int16).cpu().numpy().view(np.uint16)
    check_full(orc, inp, got, "after the timeout")
