"""GPU parity of the grouped (mixture-of-experts) GEMM, fp4_gemm_grouped, against
the CPU oracle's grouped_gemm_rows (independent per-group GEMMs).

Tolerances as the plain GEMM (tests/test_gemm_gpu.py) and, with an epilogue,
as tests/test_fused_gpu.py (the bias of each row's own group). Covered: both
plans (direct with one CTA or a CTA pair per MMA; swap-AB with N tiles 64 to
256, one or several tiles per group), empty groups, groups that are not
multiples of 128 rows, N not a multiple of the tile, plain and prepacked
weight scales, fused epilogues with per-group bias, K = 0, and the MoE
workloads at full size on sampled rows.
"""
from __future__ import annotations

import numpy as np
import pytest

import workloads as W
from tests.test_fused_gpu import check as check_fused, expected as expected_fused
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


def run_grouped(fp4, gin, act="none", bias=None, mode=0, prepacked=False, acts_prepacked=False):
    A, sfA, B, sfB = (_dev(getattr(gin, k)) for k in ("A", "sfA", "B", "sfB"))
    if prepacked:
        per = fp4.scale_atom_bytes(gin.N, gin.K, gin.vec)
        atoms = torch.empty(gin.G * per, dtype=torch.uint8, device="cuda")
        for g in range(gin.G):
            fp4.scale_reorder(sfB[g * gin.N:(g + 1) * gin.N], atoms[g * per:(g + 1) * per], gin.N, gin.K, gin.vec)
        sfB = atoms
    if acts_prepacked:
        atoms = torch.empty(max(16, fp4.scale_atom_bytes_grouped(gin.offsets, gin.K, gin.vec)), dtype=torch.uint8,
                            device="cuda")
        fp4.scale_reorder_grouped(sfA, atoms, gin.offsets, gin.K, gin.vec)
        sfA = atoms
    cols = gin.N // 2 if act == "swiglu" else gin.N
    dt = torch.float32 if gin.out == "f32" else torch.bfloat16
    D = torch.full((gin.M, cols), float("nan"), dtype=dt, device="cuda")
    b = _dev(bias) if bias is not None else None
    cfg = fp4.GemmConfig(mode=mode) if mode else None
    fp4.gemm_grouped(gin.fmt, gin.offsets, A, sfA, B, sfB, gin.alpha, D, gin.N, gin.K, gin.out, act=act, bias=b,
                     weights_prepacked=prepacked, acts_prepacked=acts_prepacked, config=cfg)
    st = fp4.get_device_status()
    assert st == fp4.FP4_OK, fp4.status_string(st)
    if gin.out == "f32":
        return D.cpu().numpy().astype(np.float64)
    return D.view(torch.int16).cpu().numpy().view(np.uint16)


def check_grouped(orc, gin, got, act="none", bias=None, rows=None, what=""):
    rows = np.arange(gin.M) if rows is None else np.asarray(rows)
    y, absd = orc.grouped_gemm_rows(gin, rows)
    if act == "none" and bias is None:
        return check_values(orc, gin.out, got[rows], y, absd, what)
    groups = np.searchsorted(gin.offsets, rows, side="right") - 1
    for g in np.unique(groups):
        sel = np.nonzero(groups == g)[0]
        bg = None if bias is None else bias.reshape(gin.G, gin.N)[g]
        ref, tol = expected_fused(orc, y[sel], absd[sel], bg, act)
        check_fused(orc, gin.out, got[rows[sel]], ref, tol, "%s group %d" % (what, g))


# fmt, out, group sizes, N, K, forced mode (0 auto, 1 direct, 2 swap-AB)
CASES = [
    ("nvfp4", "f32", [3, 0, 130, 1, 257, 64], 200, 512, 0),       # direct, one CTA per MMA
    ("mxfp4", "bf16", [300, 0, 5, 128, 129], 264, 768, 0),       # direct, CTA pairs
    ("nvfp4", "bf16", [1, 7, 0, 33, 64, 2], 300, 1024, 0),       # swap-AB, N tile 64
    ("mxfp4", "f32", [100, 200, 0, 3], 136, 512, 0),             # swap-AB, N tile 256
    ("nvfp4", "f32", [600, 10, 300], 192, 256, 2),               # swap-AB, several tiles per group
    ("nvfp4", "f32", [129, 400], 72, 256, 1),                    # direct, N below one tile
    ("nvfp4", "bf16", [0, 0, 5], 128, 4096, 0),                  # leading empty groups, long K
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "%s_%s_g%d_n%d_k%d_m%d" % (c[0], c[1], len(c[2]), c[3], c[4], c[5]))
def test_grouped_parity(fp4, orc, case):
    fmt, out, sizes, N, K, mode = case
    gin = W.make_grouped(fmt, sizes, N, K, alpha=0.5, seed=len(sizes) + N, out=out)
    check_grouped(orc, gin, run_grouped(fp4, gin, mode=mode), what=str(case))


@pytest.mark.parametrize("case", CASES[:4], ids=lambda c: "%s_%s_g%d" % (c[0], c[1], len(c[2])))
def test_grouped_prepacked_weights(fp4, orc, case):
    fmt, out, sizes, N, K, mode = case
    gin = W.make_grouped(fmt, sizes, N, K, seed=3, out=out)
    check_grouped(orc, gin, run_grouped(fp4, gin, mode=mode, prepacked=True), what="prepacked %s" % (case,))


def test_scale_reorder_grouped_bit_exact(fp4, orc):
    offsets = np.array([0, 130, 130, 131, 400, 528], np.int64)
    for K, vec in ((256, 16), (96, 32), (4096, 16)):
        ksf = K // vec
        sf = np.random.default_rng(K).integers(0, 256, (int(offsets[-1]), ksf)).astype(np.uint8)
        nbytes = fp4.scale_atom_bytes_grouped(offsets, K, vec)
        want = np.concatenate([orc.scale_reorder(sf[o0:o1], int(o1 - o0), ksf)
                               for o0, o1 in zip(offsets[:-1], offsets[1:]) if o1 > o0])
        assert nbytes == want.size
        out = torch.full((nbytes,), 0xAB, dtype=torch.uint8, device="cuda")
        fp4.scale_reorder_grouped(_dev(sf), out, offsets, K, vec)
        np.testing.assert_array_equal(out.cpu().numpy(), want)


@pytest.mark.parametrize("case", CASES[:4], ids=lambda c: "%s_%s_g%d" % (c[0], c[1], len(c[2])))
def test_grouped_both_prepacked(fp4, orc, case):
    fmt, out, sizes, N, K, mode = case
    gin = W.make_grouped(fmt, sizes, N, K, seed=13, out=out)
    got = run_grouped(fp4, gin, mode=mode, prepacked=True, acts_prepacked=True)
    check_grouped(orc, gin, got, what="both prepacked %s" % (case,))


@pytest.mark.parametrize("act", ["relu", "relu2", "swiglu"])
@pytest.mark.parametrize("mode", [1, 2], ids=["direct", "swap"])
def test_grouped_fused(fp4, orc, mode, act):
    sizes, N, K = [40, 0, 300, 7], 256, 512
    gin = W.make_grouped("nvfp4", sizes, N, K, alpha=0.75, b_std=0.3, seed=8)
    bias = W.make_bias(len(sizes) * N, std=1.0, seed=5)
    got = run_grouped(fp4, gin, act=act, bias=bias, mode=mode)
    check_grouped(orc, gin, got, act=act, bias=bias, what="fused %s mode %d" % (act, mode))


def test_grouped_matches_plain_per_group(fp4, orc):
    # each group also through the plain GEMM: both within tolerance of the oracle
    gin = W.make_grouped("mxfp4", [70, 260, 1], 320, 1024, seed=6)
    got = run_grouped(fp4, gin)
    for g in range(gin.G):
        o0, o1 = gin.offsets[g], gin.offsets[g + 1]
        if o1 == o0:
            continue
        part = W.GemmInputs("mxfp4", int(o1 - o0), gin.N, gin.K, gin.A[o0:o1], gin.sfA[o0:o1],
                            gin.B[g * gin.N:(g + 1) * gin.N], gin.sfB[g * gin.N:(g + 1) * gin.N], 1.0, "f32")
        A, sfA, B, sfB = (_dev(getattr(part, k)) for k in ("A", "sfA", "B", "sfB"))
        D = torch.empty(part.M, part.N, device="cuda")
        fp4.gemm("mxfp4", A, sfA, B, sfB, 1.0, D, part.M, part.N, part.K, "f32")
        plain = D.cpu().numpy().astype(np.float64)
        assert np.max(np.abs(plain - got[o0:o1])) <= 1e-4 * max(1e-30, np.max(np.abs(plain)))


@pytest.mark.parametrize("act", ["none", "relu2"])
def test_grouped_k_zero(fp4, orc, act):
    sizes, N = [2, 0, 3], 16
    offsets = np.array([0, 2, 2, 5], np.int64)
    bias = W.make_bias(3 * N, seed=9)
    D = torch.full((5, N), float("nan"), device="cuda")
    z = torch.zeros(16, dtype=torch.uint8, device="cuda")
    fp4.gemm_grouped("nvfp4", offsets, z, z, z, z, 1.0, D, N, 0, "f32", act=act, bias=_dev(bias))
    torch.cuda.synchronize()
    got = D.cpu().numpy()
    for g, (o0, o1) in enumerate(zip(offsets[:-1], offsets[1:])):
        ref = orc.epilogue(np.zeros((int(o1 - o0), N)), bias[g * N:(g + 1) * N], act)
        np.testing.assert_allclose(got[o0:o1], ref, rtol=1e-6, atol=1e-30)


def test_grouped_deterministic(fp4):
    gin = W.make_grouped("nvfp4", [30, 500, 0, 77], 384, 1024, seed=1)
    np.testing.assert_array_equal(run_grouped(fp4, gin), run_grouped(fp4, gin))


@pytest.mark.parametrize("name", sorted(W.GROUPED_WORKLOADS))
def test_grouped_workload_sampled(fp4, orc, name):
    gin, act = W.make_grouped_workload(name)
    got = run_grouped(fp4, gin, act=act)
    # every group's first and last row, and random rows
    rng = np.random.default_rng(3)
    ends = np.concatenate([gin.offsets[:-1][np.diff(gin.offsets) > 0], gin.offsets[1:][np.diff(gin.offsets) > 0] - 1])
    rows = np.unique(np.concatenate([ends, rng.integers(0, gin.M, 24)]))
    check_grouped(orc, gin, got, act=act, rows=rows, what=name)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_grouped_many_groups(fp4, orc, fmt):
    # 256 groups (the most one call takes), most of them empty or a few rows,
    # one large; K not a multiple of the 256-element k-tile
    rng = np.random.default_rng(21)
    sizes = np.where(rng.random(256) < 0.6, 0, rng.integers(1, 20, 256))
    sizes[77] = 300
    gin = W.make_grouped(fmt, sizes, 64, 288, seed=4)
    got = run_grouped(fp4, gin)
    rows = np.unique(np.concatenate([np.arange(0, gin.M, 7), [gin.M - 1]]))
    check_grouped(orc, gin, got, rows=rows, what="256 groups %s" % fmt)
