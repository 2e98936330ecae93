"""Calls recorded into CUDA graphs (stream capture) and replayed on new inputs.

One plain call of each kind runs first (it sets the kernels' attributes), then
the call is captured once and the graph replayed three times, each time on
fresh inputs copied into the captured buffers. Every replay is compared with
the CPU oracle (tolerances as tests/test_gemm_gpu.py, tests/test_fused_gpu.py
and tests/test_grouped_gpu.py) and bit for bit with a plain call of the same
plan on the same inputs. Covered: the split last wave (its exchange flags are
replayed with the graph), the reorder launch with its dependent GEMM launch,
split-K with the reduce kernel, CTA pairs, the narrow-M kernel, a fused
epilogue, the grouped GEMM, and the quantiser feeding the GEMM.
"""
from __future__ import annotations

import numpy as np
import pytest

import workloads as W
from tests.test_fused_gpu import check as check_fused, expected as expected_fused
from tests.test_gemm_gpu import check_full, run
from tests.test_grouped_gpu import check_grouped, run_grouped
from tests._helpers import bf16_bits_to_f64, bf16_ulp

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

REPLAYS = 3


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


def capture(call):
    """One plain call on a side stream, then the same call captured into a graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    torch.cuda.synchronize()
    return g


def replay(fp4, g):
    g.replay()
    torch.cuda.synchronize()
    st = fp4.get_device_status()
    assert st == fp4.FP4_OK, fp4.status_string(st)


# fmt, out, M, N, K, (mode, bn, cta_group, max_ctas, splits, split_tail), act
CASES = [
    ("nvfp4", "bf16", 768, 768, 1280, (1, 256, 1, 14, 0, 1), "none"),  # 18 tiles on 14 CTAs: 4 split
    ("mxfp4", "f32", 512, 1024, 1312, (1, 256, 1, 12, 0, 1), "none"),  # split last wave, K tail
    ("nvfp4", "f32", 40, 2000, 4096, (2, 64, 1, 0, 4, 0), "none"),     # swap-AB, split-K + reduce
    ("mxfp4", "bf16", 384, 640, 2048, (1, 256, 2, 10, 0, 0), "none"),  # CTA pairs
    ("nvfp4", "f32", 1, 300, 4096, (3, 0, 0, 0, 0, 0), "none"),        # narrow-M kernel
    ("nvfp4", "bf16", 768, 768, 1280, (1, 256, 1, 14, 0, 1), "swiglu"),  # fused epilogue, split last wave
]


@pytest.mark.parametrize("prepacked", [False, True], ids=["plain", "atoms"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "%s_%s_%dx%dx%d_m%d_%s" % (c[:5] + (c[5][0], c[6])))
def test_gemm_graph_replays(fp4, orc, case, prepacked):
    fmt, out, M, N, K, (mode, bn, cg, cap, splits, tail), act = case
    cfg = fp4.GemmConfig(mode=mode, bn=bn, cta_group=cg, max_ctas=cap, splits=splits, split_tail=tail)
    inps = [W.make_random(fmt, M, N, K, out=out, alpha=0.5, b_std=0.3, seed=50 + i) for i in range(REPLAYS)]
    bias = W.make_bias(N, std=1.0, seed=7) if act != "none" else None
    bufs = {k: _dev(getattr(inps[0], k)) for k in ("A", "sfA", "B", "sfB")}
    vec = inps[0].vec
    if prepacked:
        pa = torch.empty(fp4.scale_atom_bytes(M, K, vec), dtype=torch.uint8, device="cuda")
        pb = torch.empty(fp4.scale_atom_bytes(N, K, vec), dtype=torch.uint8, device="cuda")
    cols = N // 2 if act == "swiglu" else N
    dt = torch.float32 if out == "f32" else torch.bfloat16
    D = torch.full((M, cols), float("nan"), dtype=dt, device="cuda")
    b = _dev(bias) if bias is not None else None

    def load(inp):
        for k in bufs:
            bufs[k].copy_(torch.from_numpy(np.ascontiguousarray(getattr(inp, k))))
        if prepacked:
            fp4.scale_reorder(bufs["sfA"], pa, M, K, vec)
            fp4.scale_reorder(bufs["sfB"], pb, N, K, vec)

    def call():
        sfa, sfb = (pa, pb) if prepacked else (bufs["sfA"], bufs["sfB"])
        fp4.gemm_fused(fmt, bufs["A"], sfa, bufs["B"], sfb, 0.5, D, M, N, K, out, act=act, bias=b,
                       prepacked=prepacked, config=cfg)

    load(inps[0])
    g = capture(call)
    for i in (1, 2, 0):
        load(inps[i])
        D.fill_(float("nan"))
        replay(fp4, g)
        got = _host(D, out)
        what = "graph replay %d %s" % (i, case)
        if act == "none":
            check_full(orc, inps[i], got, what)
            np.testing.assert_array_equal(got, run(fp4, inps[i], cfg, prepacked=prepacked))
        else:
            y, absd = orc.gemm_rows(inps[i])
            ref, tol = expected_fused(orc, y, absd, bias, act)
            check_fused(orc, out, got, ref, tol, what)
            D2 = torch.full_like(D, float("nan"))
            load(inps[i])
            fp4.gemm_fused(fmt, bufs["A"], pa if prepacked else bufs["sfA"], bufs["B"],
                           pb if prepacked else bufs["sfB"], 0.5, D2, M, N, K, out, act=act, bias=b,
                           prepacked=prepacked, config=cfg)
            torch.cuda.synchronize()
            np.testing.assert_array_equal(got, _host(D2, out))


@pytest.mark.parametrize("mode", [1, 2], ids=["direct", "swap"])
def test_grouped_graph_replays(fp4, orc, mode):
    sizes, N, K = [40, 0, 300, 7, 129], 256, 1024
    gins = [W.make_grouped("nvfp4", sizes, N, K, alpha=0.5, seed=60 + i, out="bf16") for i in range(REPLAYS)]
    g0 = gins[0]
    bufs = {k: _dev(getattr(g0, k)) for k in ("A", "sfA", "B", "sfB")}
    D = torch.full((g0.M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    cfg = fp4.GemmConfig(mode=mode)

    def call():
        fp4.gemm_grouped("nvfp4", g0.offsets, bufs["A"], bufs["sfA"], bufs["B"], bufs["sfB"], 0.5, D, N, K, "bf16",
                         config=cfg)

    g = capture(call)
    for i in (1, 2, 0):
        gin = gins[i]
        for k in bufs:
            bufs[k].copy_(torch.from_numpy(np.ascontiguousarray(getattr(gin, k))))
        D.fill_(float("nan"))
        replay(fp4, g)
        got = _host(D, "bf16")
        check_grouped(orc, gin, got, what="grouped graph replay %d mode %d" % (i, mode))
        np.testing.assert_array_equal(got, run_grouped(fp4, gin, mode=mode))


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_quantize_then_gemm_graph(fp4, orc, fmt):
    """A layer step in one graph: quantise bf16 activations to codes and atom scales,
    then the prepacked GEMM against fixed quantised weights."""
    M, N, K = 300, 384, 2048
    vec = 16 if fmt == "nvfp4" else 32
    Xb = W.make_values(N, K, std=0.02, dtype="bf16", seed=70)
    wcodes = torch.empty(N * K // 2, dtype=torch.uint8, device="cuda")
    watoms = torch.empty(fp4.scale_atom_bytes(N, K, vec), dtype=torch.uint8, device="cuda")
    fp4.quantize(fmt, _dev(Xb.view(np.int16)), N, K, wcodes, watoms, in_dtype="bf16", layout="atom")
    X = torch.empty((M, K), dtype=torch.int16, device="cuda")
    codes = torch.empty(M * K // 2, dtype=torch.uint8, device="cuda")
    atoms = torch.empty(fp4.scale_atom_bytes(M, K, vec), dtype=torch.uint8, device="cuda")
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")

    def call():
        fp4.quantize(fmt, X, M, K, codes, atoms, in_dtype="bf16", layout="atom")
        fp4.gemm(fmt, codes, atoms, wcodes, watoms, 1.0, D, M, N, K, "bf16", prepacked=True)

    Xs = [W.make_values(M, K, dtype="bf16", seed=71 + i) for i in range(REPLAYS)]
    X.copy_(torch.from_numpy(Xs[0].view(np.int16)))
    g = capture(call)
    B, sfB = orc.quantize(Xb, fmt)
    for i in (1, 2, 0):
        X.copy_(torch.from_numpy(Xs[i].view(np.int16)))
        D.fill_(float("nan"))
        replay(fp4, g)
        got = _host(D, "bf16")
        A, sfA = orc.quantize(Xs[i], fmt)
        ref, _ = orc.gemm_rows(W.GemmInputs(fmt, M, N, K, A, sfA, B, sfB, 1.0, "bf16", "quantised"))
        refb = orc.round_bf16(ref)
        err = np.abs(bf16_bits_to_f64(got) - bf16_bits_to_f64(refb))
        assert np.all(err <= bf16_ulp(refb)), "replay %d" % i
