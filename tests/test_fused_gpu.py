"""GPU parity of the fused epilogues (fp4_gemm_fused) against the CPU oracle.

The expected values are the oracle's: its exact GEMM (fp64) followed by its
epilogue (bias, ReLU, squared ReLU, SwiGLU) in fp64. The tolerance is the
GEMM's, carried through the epilogue to first order, element by element:

  z = y + bias,   dz = 1e-5 * |alpha| * sum_k |a_k b_k| + 1e-6 + 2^-23 |z|
                  (the GEMM's fp32 bound plus the rounding of alpha * acc + bias)
  none, ReLU:     dz                      (ReLU is 1-Lipschitz)
  squared ReLU:   2 max(z, 0) dz + dz^2 + 2^-22 z^2
  SwiGLU:         1.1 dg (|u| + du) + |silu(g)| du + 2e-6 |silu(g) u|
                  (|silu'| <= 1.1; 2e-6 covers the fp32 exp, division and product)
  bf16 output:    the above plus one bf16 ulp of (|ref| + tolerance)

Plans covered: direct (one CTA per MMA, CTA pairs, the split tail), swap-AB
(with and without split-K), K = 0, ragged M and N; full-size FFN projections
on sampled rows and (row, column) pairs.
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


@pytest.fixture(scope="module")
def orc():
    import oracle
    oracle.build()
    return oracle


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_fused(fp4, inp, act, bias, cfg=None):
    """D from the device: float64 (fp32 out) or uint16 bits (bf16 out)."""
    A, sfA, B, sfB = (_dev(getattr(inp, k)) for k in ("A", "sfA", "B", "sfB"))
    cols = inp.N // 2 if act == "swiglu" else inp.N
    dt = torch.float32 if inp.out == "f32" else torch.bfloat16
    D = torch.full((inp.M, cols), float("nan"), dtype=dt, device="cuda")
    b = _dev(bias) if bias is not None else None
    fp4.gemm_fused(inp.fmt, A, sfA, B, sfB, inp.alpha, D, inp.M, inp.N, inp.K, inp.out, act=act, bias=b,
                   config=cfg)
    st = fp4.get_device_status()
    assert st == fp4.FP4_OK, fp4.status_string(st)
    if inp.out == "f32":
        return D.cpu().numpy().astype(np.float64)
    return D.view(torch.int16).cpu().numpy().view(np.uint16)


def _silu(x):
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def expected(orc, y, absd, bias, act):
    """Oracle output and its tolerance for GEMM rows y (fp64, R x C) with bounds absd;
    ``bias``: the C bias entries of y's columns, or None."""
    y = np.atleast_2d(y)
    ref = orc.epilogue(y, None if bias is None else np.ascontiguousarray(bias, dtype=np.float32), act)
    z = y + (0.0 if bias is None else np.asarray(bias, dtype=np.float64))
    dz = 1e-5 * np.atleast_2d(absd) + 1e-6 + 2.0 ** -23 * np.abs(z)
    if act in ("none", "relu"):
        tol = dz
    elif act == "relu2":
        r = np.maximum(z, 0.0)
        tol = 2.0 * r * dz + dz * dz + 2.0 ** -22 * r * r
    else:
        g, u, dg, du = z[:, 0::2], z[:, 1::2], dz[:, 0::2], dz[:, 1::2]
        s = _silu(g)
        tol = 1.1 * dg * (np.abs(u) + du) + np.abs(s) * du + 2e-6 * np.abs(s * u)
    return ref, tol


def check(orc, out, got, ref, tol, what):
    if out == "f32":
        err = np.abs(got - ref)
        lim = tol
    else:
        err = np.abs(bf16_bits_to_f64(got) - ref)
        lim = tol + bf16_ulp(orc.round_bf16(np.abs(ref) + tol))
    bad = ~(err <= lim)
    if bad.any():
        idx = tuple(np.argwhere(bad)[0])
        raise AssertionError("%s: %d/%d out of tolerance; first at %s: got %r ref %r lim %r"
                             % (what, int(bad.sum()), bad.size, idx, got[idx], ref[idx], lim[idx]))
    return float(np.max(err / np.maximum(lim, 1e-300))) if err.size else 0.0


def check_full(orc, inp, act, bias, got, what):
    y, absd = orc.gemm_rows(inp)
    ref, tol = expected(orc, y, absd, bias, act)
    return check(orc, inp.out, got, ref, tol, what)


ACTS = ["none", "relu", "relu2", "swiglu"]

# fmt, out, M, N, K, config (mode, bn, cta_group, max_ctas, splits[, split_tail]) or None
PLAN_CASES = [
    ("nvfp4", "f32", 300, 520, 512, None),                       # direct, one CTA per MMA, ragged
    ("nvfp4", "bf16", 768, 768, 1280, (1, 256, 1, 14, 0, 1)),     # direct with the split tail
    ("mxfp4", "f32", 640, 384, 768, (1, 256, 2, 0, 0)),           # direct, CTA pairs
    ("mxfp4", "bf16", 520, 272, 512, (1, 128, 2, 0, 0)),          # pairs, N tile 128
    ("nvfp4", "f32", 96, 1000, 512, None),                        # swap-AB (M <= 256)
    ("nvfp4", "bf16", 40, 2048, 4096, (2, 64, 1, 0, 3)),          # swap-AB with split-K
    ("mxfp4", "f32", 200, 602, 1024, (2, 256, 2, 0, 0)),          # swap-AB, pairs
]


def _cfg(fp4, c):
    if c is None:
        return None
    mode, bn, cg, cap, splits, *tail = c
    return fp4.GemmConfig(mode=mode, bn=bn, cta_group=cg, max_ctas=cap, splits=splits,
                          split_tail=tail[0] if tail else 0)


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("with_bias", [False, True], ids=["nobias", "bias"])
@pytest.mark.parametrize("case", PLAN_CASES, ids=lambda c: "%s_%s_%dx%dx%d" % c[:5])
def test_fused_epilogue_plans(fp4, orc, case, with_bias, act):
    fmt, out, M, N, K, c = case
    inp = W.make_random(fmt, M, N, K, out=out, alpha=0.75, a_std=1.0, b_std=0.3, seed=M + N + K)
    bias = W.make_bias(N, std=1.0, seed=N) if with_bias else None
    got = run_fused(fp4, inp, act, bias, _cfg(fp4, c))
    check_full(orc, inp, act, bias, got, "%s %s bias=%s" % (case, act, with_bias))


def test_fused_none_equals_plain_gemm(fp4, orc):
    # no bias, no activation: bit-identical to fp4_gemm on every plan
    for M, c in ((300, None), (40, (2, 64, 1, 0, 3)), (300, (1, 256, 2, 0, 0))):
        inp = W.make_random("nvfp4", M, 520, 512, out="f32", alpha=0.5, seed=3)
        A, sfA, B, sfB = (_dev(getattr(inp, k)) for k in ("A", "sfA", "B", "sfB"))
        D0 = torch.empty(inp.M, inp.N, dtype=torch.float32, device="cuda")
        D1 = torch.empty_like(D0)
        fp4.gemm(inp.fmt, A, sfA, B, sfB, inp.alpha, D0, inp.M, inp.N, inp.K, "f32", config=_cfg(fp4, c))
        fp4.gemm_fused(inp.fmt, A, sfA, B, sfB, inp.alpha, D1, inp.M, inp.N, inp.K, "f32", act="none",
                       config=_cfg(fp4, c))
        assert torch.equal(D0, D1), c


@pytest.mark.parametrize("act", ACTS)
def test_fused_k_zero(fp4, orc, act):
    # K = 0: D = epilogue(bias) on every row
    M, N = 5, 24
    bias = W.make_bias(N, std=2.0, seed=1)
    dbias = _dev(bias)
    cols = N // 2 if act == "swiglu" else N
    D = torch.full((M, cols), float("nan"), dtype=torch.float32, device="cuda")
    e = torch.empty(16, dtype=torch.uint8, device="cuda")
    fp4.gemm_fused("nvfp4", e, e, e, e, 1.0, D, M, N, 0, "f32", act=act, bias=dbias)
    ref = orc.epilogue(np.zeros((M, N)), bias, act)
    np.testing.assert_allclose(D.cpu().numpy(), ref, rtol=2e-6, atol=1e-30)


def test_fused_deterministic(fp4):
    inp = W.make_random("nvfp4", 768, 768, 1280, out="bf16", alpha=0.5, seed=11)
    bias = W.make_bias(768, seed=2)
    cfg = (1, 256, 1, 14, 0)
    a = run_fused(fp4, inp, "swiglu", bias, _cfg(fp4, cfg))
    np.testing.assert_array_equal(a, run_fused(fp4, inp, "swiglu", bias, _cfg(fp4, cfg)))


def test_swiglu_rejects_odd_n(fp4):
    inp = W.make_random("nvfp4", 8, 30, 64, seed=1)
    with pytest.raises(fp4.Fp4Error) as e:
        run_fused(fp4, W.make_random("nvfp4", 8, 31, 64, seed=1), "swiglu", None)
    assert e.value.status == 2
    run_fused(fp4, inp, "swiglu", None)


# ---- the named FFN workloads at full size, sampled ------------------------------------------

@pytest.mark.parametrize("name", sorted(W.FUSED_WORKLOADS))
def test_fused_workload_sampled(fp4, orc, name):
    inp, act, bias = W.make_fused(name)
    got = run_fused(fp4, inp, act, bias)
    glu = act == "swiglu"
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, inp.M - 1], rng.integers(0, inp.M, 6)]))
    y, absd = orc.gemm_rows(inp, rows)
    ref, tol = expected(orc, y, absd, bias, act)
    check(orc, inp.out, got[rows], ref, tol, "%s rows" % name)
    # sampled (row, D column) pairs over the whole output
    cols = inp.N // 2 if glu else inp.N
    ii = rng.integers(0, inp.M, 3000)
    jj = rng.integers(0, cols, 3000)
    ii[:3], jj[:3] = [inp.M - 1, 0, inp.M - 1], [cols - 1, cols - 1, 0]
    if glu:
        gi, gj = np.repeat(ii, 2), np.stack([2 * jj, 2 * jj + 1], 1).reshape(-1)
    else:
        gi, gj = ii, jj
    yp, ap = orc.gemm_pairs(inp, gi, gj)
    per = 2 if glu else 1
    yp, ap = yp.reshape(-1, per), ap.reshape(-1, per)
    bsel = None if bias is None else bias[gj].reshape(-1, per)
    # each pair is a one-row problem: its own bias entries
    refs, tols = [], []
    for k in range(ii.size):
        r, t = expected(orc, yp[k:k + 1], ap[k:k + 1], None if bsel is None else bsel[k], act)
        refs.append(r[0, 0])
        tols.append(t[0, 0])
    check(orc, inp.out, got[ii, jj], np.array(refs), np.array(tols), "%s pairs" % name)
