"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Tolerances (written here, applied element by element):
  fp32 output: |D - ref| <= 1e-5 * |alpha| * sum_k |a_k b_k| + 1e-6
  bf16 output: |D - bf16(ref)| <= 1 ulp of bf16(ref)
  scale reorder: bit-exact.
Small problems are compared in full; the named workloads at full size on
sampled rows (every column of each, tile edges and the last row included) and
on sampled (row, column) pairs.
"""
from __future__ import annotations

import numpy as np
import pytest

import workloads as W
from tests._helpers import bf16_bits_to_f64, bf16_ulp, parse_worked_examples

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


def run(fp4, inp, cfg=None, prepacked=False, out_buf=None):
    """Runs the GEMM on the device; returns D as float64 (fp32 out) or uint16 bits (bf16 out)."""
    A, sfA, B, sfB = (_dev(getattr(inp, k)) for k in ("A", "sfA", "B", "sfB"))
    if prepacked:
        vec = inp.vec
        pa = torch.empty(fp4.scale_atom_bytes(inp.M, inp.K, vec), dtype=torch.uint8, device="cuda")
        pb = torch.empty(fp4.scale_atom_bytes(inp.N, inp.K, vec), dtype=torch.uint8, device="cuda")
        fp4.scale_reorder(sfA, pa, inp.M, inp.K, vec)
        fp4.scale_reorder(sfB, pb, inp.N, inp.K, vec)
        sfA, sfB = pa, pb
    dt = torch.float32 if inp.out == "f32" else torch.bfloat16
    D = out_buf if out_buf is not None else torch.full((inp.M, inp.N), float("nan"), dtype=dt, device="cuda")
    fp4.gemm(inp.fmt, A, sfA, B, sfB, inp.alpha, D, inp.M, inp.N, inp.K, inp.out, prepacked=prepacked,
             config=cfg)
    st = fp4.get_device_status()
    assert st == fp4.FP4_OK, fp4.status_string(st)
    if inp.out == "f32":
        return D.cpu().numpy().astype(np.float64)
    return D.view(torch.int16).cpu().numpy().view(np.uint16)


def check_values(orc, out, got, ref, absd, what=""):
    """got / ref / absd of the same shape; raises with the first offending element."""
    if out == "f32":
        err = np.abs(got - ref)
        tol = 1e-5 * absd + 1e-6
        bad = ~(err <= tol)
    else:
        refb = orc.round_bf16(ref)
        err = np.abs(bf16_bits_to_f64(got) - bf16_bits_to_f64(refb))
        tol = bf16_ulp(refb)
        bad = ~(err <= tol)
    if bad.any():
        idx = tuple(np.argwhere(bad)[0])
        raise AssertionError("%s: %d/%d elements out of tolerance; first at %s: got %r ref %r tol %r"
                             % (what, int(bad.sum()), bad.size, idx, got[idx], ref[idx], tol[idx]))
    return float(np.max(err / np.maximum(tol, 1e-300))) if err.size else 0.0


def check_full(orc, inp, got, what=""):
    ref, absd = orc.gemm_rows(inp)
    return check_values(orc, inp.out, got, ref, absd, what or inp.name)


def sample_rows(M, n_random=8, seed=0, tile=128):
    rng = np.random.default_rng(seed)
    rows = {0, 1, M - 1, M - 2}
    for edge in range(tile, M, tile * max(1, (M // tile) // 4)):
        rows.update({edge - 1, edge})
    rows.update(rng.integers(0, M, n_random).tolist())
    return np.array(sorted(r for r in rows if 0 <= r < M), dtype=np.int64)


def check_sampled(orc, inp, got, seed=0, n_random=8, n_pairs=4000):
    rows = sample_rows(inp.M, n_random, seed)
    ref, absd = orc.gemm_rows(inp, rows)
    r1 = check_values(orc, inp.out, got[rows], ref, absd, "%s rows" % inp.name)
    rng = np.random.default_rng(seed + 1)
    ii = rng.integers(0, inp.M, n_pairs)
    jj = rng.integers(0, inp.N, n_pairs)
    ii[:4] = [inp.M - 1, inp.M - 1, 0, inp.M // 2]
    jj[:4] = [inp.N - 1, 0, inp.N - 1, inp.N - 1]
    refp, absp = orc.gemm_pairs(inp, ii, jj)
    r2 = check_values(orc, inp.out, got[ii, jj], refp, absp, "%s pairs" % inp.name)
    return max(r1, r2)


# ---- scale reorder ------------------------------------------------------------------

@pytest.mark.parametrize("ra,rb,K,vec", [(300, 1000, 288, 16), (1, 129, 4096, 16), (0, 77, 96, 32), (64, 0, 64, 32)])
def test_scale_reorder2_bit_exact(fp4, orc, ra, rb, K, vec):
    # both operands in one launch: each equal to the oracle's reorder
    rng = np.random.default_rng(ra + rb + K)
    sa = rng.integers(0, 256, (ra, K // vec)).astype(np.uint8)
    sb = rng.integers(0, 256, (rb, K // vec)).astype(np.uint8)
    na, nb = fp4.scale_atom_bytes(ra, K, vec), fp4.scale_atom_bytes(rb, K, vec)
    oa = torch.full((max(na, 16),), 0xCD, dtype=torch.uint8, device="cuda")
    ob = torch.full((max(nb, 16),), 0xCD, dtype=torch.uint8, device="cuda")
    fp4.scale_reorder2(_dev(sa) if ra else None, oa, ra, _dev(sb) if rb else None, ob, rb, K, vec)
    torch.cuda.synchronize()
    if ra:
        np.testing.assert_array_equal(oa.cpu().numpy()[:na], orc.scale_reorder(sa, ra, K // vec))
    if rb:
        np.testing.assert_array_equal(ob.cpu().numpy()[:nb], orc.scale_reorder(sb, rb, K // vec))


@pytest.mark.parametrize("rows,K,vec", [(128, 64, 16), (300, 288, 16), (1, 32, 32), (257, 4096, 16),
                                        (1000, 96, 32), (14336, 4096, 16), (129, 5120, 32)])
def test_scale_reorder_bit_exact(fp4, orc, rows, K, vec):
    rng = np.random.default_rng(rows + K)
    sf = rng.integers(0, 256, (rows, K // vec)).astype(np.uint8)
    nbytes = fp4.scale_atom_bytes(rows, K, vec)
    assert nbytes == orc.scale_atom_bytes(rows, K // vec)
    out = torch.full((nbytes,), 0xAB, dtype=torch.uint8, device="cuda")   # padding must be written
    fp4.scale_reorder(_dev(sf), out, rows, K, vec)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy(), orc.scale_reorder(sf, rows, K // vec))


def test_scale_reorder_unaligned_source(fp4, orc):
    # plain scales need no alignment: an odd source address takes the byte path
    rows, K, vec = 200, 1024, 16
    sf = np.random.default_rng(1).integers(0, 256, (rows, K // vec)).astype(np.uint8)
    buf = torch.zeros(sf.size + 16, dtype=torch.uint8, device="cuda")
    buf[1:1 + sf.size] = _dev(sf.ravel())
    out = torch.empty(fp4.scale_atom_bytes(rows, K, vec), dtype=torch.uint8, device="cuda")
    fp4.scale_reorder(buf.data_ptr() + 1, out, rows, K, vec)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy(), orc.scale_reorder(sf, rows, K // vec))


# ---- small problems, full comparison -------------------------------------------------------

def test_smallest_config_matches(fp4, orc):
    inp = W.make_config("nvfp4_128x128x256_f32")
    check_full(orc, inp, run(fp4, inp))


def test_worked_examples(fp4, orc):
    for inp, D in parse_worked_examples():
        got = run(fp4, inp)
        np.testing.assert_array_equal(got, D, err_msg=inp.name)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_one_hot_products_exact(fp4, orc, fmt):
    # one nonzero code per row: every output is 0 or a single exact product,
    # so any permutation of rows, k or scale bytes shows up as a mismatch
    rng = np.random.default_rng(3)
    M, N, K = 256, 256, 1024
    vec = 16 if fmt == "nvfp4" else 32
    ka = rng.integers(0, K, M)
    kb = ka[rng.integers(0, M, N)]
    kb[::3] = rng.integers(0, K, kb[::3].size)
    codes_a = np.zeros((M, K), np.uint8)
    codes_b = np.zeros((N, K), np.uint8)
    codes_a[np.arange(M), ka] = rng.integers(1, 16, M)
    codes_b[np.arange(N), kb] = rng.integers(1, 16, N)
    lo, hi = (0x20, 0x60) if fmt == "nvfp4" else (118, 138)
    sfA = rng.integers(lo, hi, (M, K // vec)).astype(np.uint8)
    sfB = rng.integers(lo, hi, (N, K // vec)).astype(np.uint8)
    inp = W.GemmInputs(fmt, M, N, K, W.pack_codes(codes_a), sfA, W.pack_codes(codes_b), sfB, 1.0, "f32", "onehot")
    ref, _ = orc.gemm_rows(inp)
    plans = [None,
             fp4.GemmConfig(mode=1, bn=256, cta_group=1), fp4.GemmConfig(mode=1, bn=128, cta_group=1),
             fp4.GemmConfig(mode=1, bn=256, cta_group=2), fp4.GemmConfig(mode=1, bn=128, cta_group=2),
             fp4.GemmConfig(mode=2, bn=256, cta_group=1), fp4.GemmConfig(mode=2, bn=256, cta_group=2)]
    for cfg in plans:
        got = run(fp4, inp, cfg)
        what = "auto" if cfg is None else (cfg.mode, cfg.bn, cfg.cta_group)
        np.testing.assert_array_equal(got, ref, err_msg=str(what))


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_uniform_codes_several_tiles(fp4, orc, fmt, out):
    inp = W.make_uniform_codes(fmt, 384, 640, 1280, out=out, alpha=0.75, seed=11)
    check_full(orc, inp, run(fp4, inp))


PLAN_CASES = [
    # (mode, bn, splits, cta_group): direct and swap-AB, both tile widths, one CTA
    # or a CTA pair per MMA, split-K
    (1, 256, 0, 1), (1, 128, 0, 1), (1, 256, 0, 2), (1, 128, 0, 2), (2, 256, 0, 1), (2, 128, 0, 1),
    (2, 256, 0, 2), (2, 128, 2, 2), (2, 128, 3, 1), (2, 128, 2, 1), (2, 256, 3, 2), (1, 256, 0, 2),
    (1, 64, 0, 1), (1, 32, 0, 1),
]


@pytest.mark.parametrize("seed", range(24))
def test_fuzz_small_shapes(fp4, orc, seed):
    rng = np.random.default_rng(1000 + seed)
    fmt = ["nvfp4", "mxfp4"][seed % 2]
    out = ["f32", "bf16"][(seed // 2) % 2]
    M = int(rng.integers(1, 301))
    N = int(rng.integers(1, 301))
    if out == "bf16":
        N += (-N) % 8 if seed % 3 else 0       # aligned rows for TMA stores half the time
    K = int(rng.integers(1, 33)) * 32
    dist = "t3" if seed % 3 == 0 else "normal"
    inp = W.make_random(fmt, M, N, K, dist=dist, alpha=float(rng.choice([1.0, 0.5, 3.0])), out=out, seed=seed)
    check_full(orc, inp, run(fp4, inp), "auto plan")
    mode, bn, splits, cg = PLAN_CASES[seed % len(PLAN_CASES)]
    esize = 4 if out == "f32" else 2
    rows_b = N if mode == 1 else M
    if mode == 1 and (N * esize) % 16:
        mode = 2
        rows_b = M
    if rows_b > bn and bn < 128:
        bn = 256
    cfg = fp4.GemmConfig(mode=mode, bn=bn, splits=splits, cta_group=cg)
    check_full(orc, inp, run(fp4, inp, cfg), "plan %s" % ((mode, bn, splits, cg),))


@pytest.mark.parametrize("M", [1, 7, 16, 33, 64, 100, 128, 200, 256])
def test_skinny_swap_widths(fp4, orc, M):
    inp = W.make_random("nvfp4", M, 1000, 512, out="bf16", seed=M)
    check_full(orc, inp, run(fp4, inp))
    check_full(orc, inp, run(fp4, inp, fp4.GemmConfig(mode=2, splits=2)), "split 2")


# Swap-AB tiles of CTA pairs leave through TMA boxes of 32 D columns x 64 (bf16)
# or 32 (fp32) D rows: ragged D edges on both axes, both output types, N tiles of
# 128 and 256, and D rows whose pitch is not a multiple of 16 bytes (the direct
# stores instead).
TRANSPOSED_CASES = [("nvfp4", "bf16", 200, 1000, 512, 256), ("nvfp4", "f32", 130, 4112, 768, 256),
                    ("mxfp4", "bf16", 100, 600, 1024, 128), ("mxfp4", "f32", 77, 2056, 512, 128),
                    ("nvfp4", "f32", 250, 1001, 256, 256)]


@pytest.mark.parametrize("fmt,out,M,N,K,bn", TRANSPOSED_CASES)
def test_swap_pairs_tma_box_edges(fp4, orc, fmt, out, M, N, K, bn):
    inp = W.make_random(fmt, M, N, K, out=out, seed=M + N)
    cfg = fp4.GemmConfig(mode=2, bn=bn, cta_group=2)
    assert fp4.gemm_plan(fmt, M, N, K, out, config=cfg)["cta_group"] == 2
    check_full(orc, inp, run(fp4, inp, cfg), "swap pair %s" % ((fmt, out, M, N, K, bn),))


def test_k_tail_not_multiple_of_tile(fp4, orc):
    for K in (32, 96, 288, 544, 800):
        for fmt in ("nvfp4", "mxfp4"):
            inp = W.make_random(fmt, 130, 136, K, out="f32", seed=K)
            check_full(orc, inp, run(fp4, inp), "K=%d %s" % (K, fmt))
            check_full(orc, inp, run(fp4, inp, fp4.GemmConfig(mode=2, bn=256)), "K=%d %s swap" % (K, fmt))
            check_full(orc, inp, run(fp4, inp, fp4.GemmConfig(mode=1, bn=128, cta_group=2)),
                       "K=%d %s pair" % (K, fmt))


@pytest.mark.parametrize("K", [256, 768, 1280, 1792])
def test_mxfp4_pairs_k_lengths(fp4, orc, K):
    # CTA pairs over odd and even k-tile counts, direct and split-K
    inp = W.make_random("mxfp4", 520, 384, K, out="bf16", seed=K)
    check_full(orc, inp, run(fp4, inp, fp4.GemmConfig(mode=1, bn=256, cta_group=2)), "direct K=%d" % K)
    check_full(orc, inp, run(fp4, inp, fp4.GemmConfig(mode=1, bn=128, cta_group=2)), "direct bn128 K=%d" % K)
    check_full(orc, inp, run(fp4, inp, fp4.GemmConfig(mode=2, bn=256, cta_group=2, splits=3)), "split K=%d" % K)


@pytest.mark.parametrize("M,N,K,bn,splits", [(40, 2000, 4096, 64, 4), (16, 300, 14336, 16, 7), (100, 640, 2048, 128, 5),
                                              (200, 136, 1024, 256, 3)])
def test_split_k_plans(fp4, orc, M, N, K, bn, splits):
    # forced K splits over tile widths 16 .. 256 (fixed summation order)
    inp = W.make_random("nvfp4", M, N, K, out="f32", seed=M + splits)
    cfg = fp4.GemmConfig(mode=2, bn=bn, splits=splits, cta_group=2 if bn == 256 else 1)
    a = run(fp4, inp, cfg)
    check_full(orc, inp, a, "split-K %s" % ((M, N, K, bn, splits),))
    np.testing.assert_array_equal(a, run(fp4, inp, cfg))


@pytest.mark.parametrize("M,N,K,cfg", [(300, 520, 1024, None), (768, 768, 1280, (1, 256, 1)), (40, 1000, 2048, (2, 64, 1)),
                                       (16, 700, 4096, (2, 16, 1)), (200, 384, 768, (2, 256, 1)),
                                       (129, 264, 512, (1, 128, 1)), (300, 520, 1056, None)])
def test_nvfp4_plain_equals_prepacked(fp4, orc, M, N, K, cfg):
    # plain NVFP4 scales (reordered by the call) against the prepacked call on the
    # same plan: bit-identical, and within tolerance of the oracle
    inp = W.make_random("nvfp4", M, N, K, out="f32", alpha=0.5, dist="t3", seed=M + K)
    c = None if cfg is None else fp4.GemmConfig(mode=cfg[0], bn=cfg[1], cta_group=cfg[2])
    plan = fp4.gemm_plan("nvfp4", M, N, K, "f32", config=c)
    assert plan["launches"] == 2 + (1 if plan["splits"] > 1 else 0)
    a = run(fp4, inp, c)
    check_full(orc, inp, a, "plain scales %s" % ((M, N, K, cfg),))
    np.testing.assert_array_equal(a, run(fp4, inp, c, prepacked=True))


def test_nvfp4_plain_scales_unaligned(fp4, orc):
    # scales at an address that is not 16-byte aligned (the reorder reads bytes)
    inp = W.make_random("nvfp4", 300, 256, 512, out="f32", seed=2)
    A, sfA, B, sfB = (_dev(getattr(inp, k)) for k in ("A", "sfA", "B", "sfB"))
    buf = torch.zeros(inp.sfA.size + 4, dtype=torch.uint8, device="cuda")
    buf[4:] = torch.from_numpy(inp.sfA.reshape(-1)).cuda()
    D = torch.full((inp.M, inp.N), float("nan"), device="cuda")
    fp4.gemm("nvfp4", A, buf.data_ptr() + 4, B, sfB, inp.alpha, D, inp.M, inp.N, inp.K, "f32")
    assert fp4.get_device_status() == fp4.FP4_OK
    check_full(orc, inp, D.cpu().numpy().astype(np.float64), "unaligned scales")


def test_prepacked_equals_plain(fp4, orc):
    inp = W.make_random("mxfp4", 300, 520, 768, out="f32", seed=4)
    a = run(fp4, inp)
    b = run(fp4, inp, prepacked=True)
    np.testing.assert_array_equal(a, b)


def test_deterministic_bytes(fp4, orc):
    inp = W.make_random("nvfp4", 700, 1100, 2048, out="bf16", seed=5)
    a = run(fp4, inp)
    b = run(fp4, inp)
    np.testing.assert_array_equal(a, b)
    c = run(fp4, inp, fp4.GemmConfig(mode=2, splits=4))
    d = run(fp4, inp, fp4.GemmConfig(mode=2, splits=4))
    np.testing.assert_array_equal(c, d)


# Asked for (split_tail = 1), the last, partial wave of direct-mode tiles runs as
# two K halves when it fills at most half of the resident CTAs or CTA pairs (the
# caps below force such tails).
SPLIT_TAIL_CASES = [
    # fmt, out, M, N, K, (mode, bn, cta_group, max_ctas)
    ("nvfp4", "bf16", 768, 768, 1280, (1, 256, 1, 14)),     # 18 tiles on 14 CTAs: 4 split, odd k-tile count
    ("mxfp4", "f32", 768, 768, 1280, (1, 256, 1, 14)),
    ("nvfp4", "f32", 512, 1024, 1312, (1, 256, 1, 12)),     # 16 tiles on 12 CTAs: 4 split; K tail
    ("mxfp4", "bf16", 384, 640, 2048, (1, 256, 1, 6)),      # 9 tiles on 6 CTAs: 3 split; partial tiles
    ("nvfp4", "f32", 256, 256, 1024, (1, 256, 1, 0)),       # 2 tiles, every CTA free: both split
    # CTA pairs (tiles of 256 x 256; each CTA of a pair parks and adds its own rows)
    ("nvfp4", "bf16", 384, 640, 2048, (1, 256, 2, 10)),     # 6 pair tiles on 5 pairs: 1 split; partial tiles
    ("nvfp4", "bf16", 1024, 768, 1280, (1, 256, 2, 20)),    # 12 on 10 pairs: 2 split, odd k-tile count
    ("mxfp4", "f32", 640, 640, 2048, (1, 256, 2, 16)),      # 9 on 8 pairs: 1 split; partial tiles
    ("nvfp4", "f32", 512, 1024, 1312, (1, 256, 2, 12)),     # 8 on 6 pairs: 2 split; K tail
    ("mxfp4", "bf16", 512, 512, 1024, (1, 256, 2, 0)),      # 4 pair tiles, every pair free: all split
]


@pytest.mark.parametrize("case", SPLIT_TAIL_CASES, ids=lambda c: "%s_%s_%dx%dx%d" % c[:5])
def test_split_tail(fp4, orc, case):
    fmt, out, M, N, K, (mode, bn, cg, cap) = case
    inp = W.make_random(fmt, M, N, K, out=out, alpha=0.5, seed=M + K)
    cfg = fp4.GemmConfig(mode=mode, bn=bn, cta_group=cg, max_ctas=cap, split_tail=1)
    a = run(fp4, inp, cfg)
    check_full(orc, inp, a, "split tail %s" % (case,))
    np.testing.assert_array_equal(a, run(fp4, inp, cfg))      # fixed summation order


# The automatic plan on skinny and few-tile shapes, as measured fastest on GB300
# (152 SMs) with forced plans: (M, N, K) -> (swap, N tile, CTA group, K splits).
PLAN_CHOICES = [
    ((16, 4096, 14336), (True, 16, 1, 4)),      # long K, few tiles: split K
    ((64, 4096, 28672), (True, 64, 1, 4)),
    ((16, 14336, 4096), (True, 16, 1, 1)),      # enough tiles: one pass
    ((128, 4096, 14336), (True, 128, 2, 1)),    # a split's reduce costs more than it saves
    ((128, 2048, 8192), (True, 128, 2, 1)),
    ((256, 4096, 14336), (False, 128, 2, 1)),   # few pair tiles: direct, N tiles of 128
    ((512, 2048, 8192), (False, 128, 2, 1)),
    ((1024, 14336, 4096), (False, 256, 2, 1)),  # enough tiles: N tiles of 256
    ((8192, 8192, 8192), (False, 256, 2, 1)),
]


@pytest.mark.parametrize("shape,want", PLAN_CHOICES, ids=lambda v: "x".join(map(str, v)) if len(v) == 3 else None)
def test_automatic_plan_choices(fp4, shape, want):
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the choices were measured on a 152-SM GB300")
    M, N, K = shape
    p = fp4.gemm_plan("nvfp4", M, N, K, "bf16", prepacked=True)
    assert (p["swap"], p["bn"], p["cta_group"], p["splits"]) == want, p


def test_persistent_grid_cap(fp4, orc):
    # few CTAs, many tiles each: exercises the stage / accumulator phase wrap-around
    inp = W.make_random("nvfp4", 1024, 1024, 1024, out="f32", seed=6)
    for cfg in (fp4.GemmConfig(max_ctas=3), fp4.GemmConfig(mode=2, bn=128, max_ctas=2),
                fp4.GemmConfig(mode=1, bn=128, max_ctas=1, cta_group=1),
                fp4.GemmConfig(mode=1, bn=256, max_ctas=2, cta_group=2),
                fp4.GemmConfig(mode=2, bn=128, max_ctas=4, cta_group=2, splits=3)):
        check_full(orc, inp, run(fp4, inp, cfg), "cap")


def test_repeated_calls_full_size(fp4, orc):
    # 8192^3 NVFP4 with CTA pairs: five stages, ~14 units per pair.
    # Timing-dependent protocol faults (a parity wait that misses its phase shows
    # up as a bounded wait running out) need several calls under load to show:
    # each repeated call must end with the status clear and give the same bytes.
    inp = W.make_config("nvfp4_8192_f32")
    A, sfA, B, sfB = (_dev(getattr(inp, k)) for k in ("A", "sfA", "B", "sfB"))
    D = torch.empty(inp.M, inp.N, dtype=torch.float32, device="cuda")
    first = None
    for _ in range(4):
        fp4.gemm(inp.fmt, A, sfA, B, sfB, inp.alpha, D, inp.M, inp.N, inp.K, inp.out)
        st = fp4.get_device_status()
        assert st == fp4.FP4_OK, fp4.status_string(st)
        got = D.cpu().numpy()
        if first is None:
            first = got.copy()
        else:
            np.testing.assert_array_equal(got, first)
    check_sampled(orc, inp, first.astype(np.float64), n_random=4)


# ---- the named workloads at full size, sampled -------------------------------------------

SAMPLED = [n for n in W.config_names() if n != "nvfp4_128x128x256_f32"]


@pytest.mark.parametrize("name", SAMPLED)
def test_named_workload_sampled(fp4, orc, name):
    inp = W.make_config(name)
    got = run(fp4, inp)
    assert np.isfinite(got).all() if inp.out == "f32" else True
    check_sampled(orc, inp, got, n_random=4 if inp.M * inp.N * inp.K > 2 ** 36 else 8)


# ---- the host-buffer path, empty and degenerate calls -----------------------------------------

def test_host_buffers(fp4, orc):
    inp = W.make_random("nvfp4", 200, 264, 640, out="bf16", seed=8)
    D = np.full((inp.M, inp.N), 0x7FC0, np.uint16)
    A, sfA, B, sfB = (np.ascontiguousarray(getattr(inp, k)) for k in ("A", "sfA", "B", "sfB"))
    fp4.gemm_host(inp.fmt, A, sfA, B, sfB, inp.alpha, D, inp.M, inp.N, inp.K, inp.out)
    torch.cuda.synchronize()
    check_full(orc, inp, D)


def test_empty_and_k_zero(fp4):
    D = torch.full((4, 8), 7.0, device="cuda")
    z = torch.zeros(16, dtype=torch.uint8, device="cuda")
    assert fp4.gemm("nvfp4", z, z, z, z, 1.0, D, 0, 8, 64, "f32") == 0
    assert fp4.gemm("nvfp4", z, z, z, z, 1.0, D, 4, 0, 64, "f32") == 0
    torch.cuda.synchronize()
    assert (D == 7.0).all()
    fp4.gemm("nvfp4", None, None, None, None, 1.0, D, 4, 8, 0, "f32")
    torch.cuda.synchronize()
    assert (D == 0.0).all()


def test_error_statuses_launch_nothing(fp4):
    z = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    D = torch.zeros(64, 64, device="cuda")
    g = lambda *a, **k: fp4.gemm(*a, check=False, **k)
    assert g("nvfp4", z, z, z, z, 1.0, D, 64, 64, 48, "f32") == 2            # K % 32
    assert g("nvfp4", z, z, z, z, 1.0, D, -1, 64, 64, "f32") == 1
    assert g("nvfp4", None, z, z, z, 1.0, D, 64, 64, 64, "f32") == 1
    assert g("nvfp4", z[1:], z, z, z, 1.0, D, 64, 64, 64, "f32") == 3         # misaligned A
    assert g("nvfp4", z, z, z, z, 1.0, D, 64, 300, 64, "f32", config=fp4.GemmConfig(mode=1, bn=64)) == 2
    assert g("nvfp4", z, z, z, z, 1.0, D, 64, 64, 64, "f32", config=fp4.GemmConfig(mode=1, splits=2)) == 2
    assert g("nvfp4", z, z, z, z, 1.0, D, 64, 64, 64, "f32", config=fp4.GemmConfig(bn=48)) == 1
    assert g("nvfp4", z, z, z, z, 1.0, D, 64, 64, 64, "f32", config=fp4.GemmConfig(cta_group=3)) == 1
    assert g("nvfp4", z, z, z, z, 1.0, D, 64, 64, 64, "f32", config=fp4.GemmConfig(bn=64, cta_group=2)) == 2
    assert fp4.get_device_status() == 0


def test_two_host_threads_two_streams(fp4, orc):
    # calls from two host threads on their own streams, first use of several
    # kernel variants racing: every result matches the oracle
    import threading
    cases = [W.make_random("nvfp4", 300, 520, 512, out="f32", seed=31),
             W.make_random("mxfp4", 64, 777, 1024, out="bf16", seed=32)]
    refs = [orc.gemm_rows(inp) for inp in cases]
    results, errors = {}, []

    def worker(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for rep in range(3):
                    results[(i, rep)] = run(fp4, cases[i], None)
        except Exception as e:          # reported below
            errors.append(repr(e))

    ts = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in ts:
        t.start()
    for t in ts:
        t.join(120)
    assert not errors, errors
    for (i, rep), got in results.items():
        ref, absd = refs[i]
        check_values(orc, cases[i].out, got, ref, absd, "thread %d rep %d" % (i, rep))
