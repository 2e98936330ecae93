"""GPU parity of the quantisation kernel (fp4_quantize) against the CPU oracle.

The bar is bit-exact: every code byte and every scale byte, in both scale
layouts, for fp32 and bf16 inputs; guard bytes past each output must stay
untouched. Cases: ragged shapes (rows not a multiple of 128, scale columns not
a multiple of 4), every finite bf16 bit pattern, exact E2M1 and E4M3 ties and
their neighbours, zero / negative-zero / subnormal / saturating blocks, the
named activation workloads at full size, and the quantiser feeding the GEMM.
"""
from __future__ import annotations

import numpy as np
import pytest

import workloads as W
from tests._helpers import bf16_bits_to_f64, bf16_ulp, torch_scale_values

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

GUARD = 64


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


def vec_of(fmt):
    return 16 if fmt == "nvfp4" else 32


def run_quant(fp4, X, fmt, layout="plain", stream=None):
    """Quantises host X (float32 or uint16 bf16 bits) on the device; returns (codes, sf) as numpy."""
    rows, K = X.shape
    in_dtype = "bf16" if X.dtype == np.uint16 else "f32"
    src = X.view(np.int16) if X.dtype == np.uint16 else X
    Xd = torch.from_numpy(np.ascontiguousarray(src)).cuda()
    n_codes = rows * K // 2
    n_sf = rows * (K // vec_of(fmt)) if layout == "plain" else fp4.scale_atom_bytes(rows, K, vec_of(fmt))
    codes = torch.full((n_codes + GUARD,), 0xAB, dtype=torch.uint8, device="cuda")
    sf = torch.full((n_sf + GUARD,), 0xCD, dtype=torch.uint8, device="cuda")
    fp4.quantize(fmt, Xd, rows, K, codes, sf, in_dtype=in_dtype, layout=layout, stream=stream)
    st = fp4.get_device_status(stream)
    assert st == fp4.FP4_OK, fp4.status_string(st)
    c = codes.cpu().numpy()
    s = sf.cpu().numpy()
    assert np.all(c[n_codes:] == 0xAB), "codes written past the end"
    assert np.all(s[n_sf:] == 0xCD), "scales written past the end"
    return c[:n_codes].reshape(rows, K // 2), s[:n_sf]


def expect(orc, X, fmt, layout):
    codes, sf = orc.quantize(X, fmt)
    if layout == "atom":
        rows, K = X.shape
        sf = orc.scale_reorder(sf, rows, K // vec_of(fmt))
    else:
        sf = sf.reshape(-1)
    return codes, sf


def assert_same(got, want, what):
    if not np.array_equal(got, want):
        bad = np.argwhere(np.asarray(got) != np.asarray(want))
        i = tuple(bad[0])
        raise AssertionError("%s: %d bytes differ; first at %s: got %#x want %#x"
                             % (what, len(bad), i, int(got[i]), int(want[i])))


def check(fp4, orc, X, fmt, layout, what=""):
    got_c, got_s = run_quant(fp4, X, fmt, layout)
    want_c, want_s = expect(orc, X, fmt, layout)
    assert_same(got_c, want_c, "codes " + what)
    assert_same(got_s, want_s, "scales " + what)


# rows: one partial band, whole bands, a partial second band, a chunk of two
# bands followed by a partial one, 256-row chunks with a band wholly past the
# matrix; K: whole and partial 4-block chunk columns in both formats
SHAPES = [(1, 32), (128, 64), (129, 96), (300, 1024), (257, 4128), (64, 32), (384, 1056), (511, 544)]


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("layout", ["plain", "atom"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "%dx%d" % s)
def test_matches_oracle(fp4, orc, fmt, dtype, layout, shape):
    rows, K = shape
    X = W.make_values(rows, K, dist="t3", std=0.5, dtype=dtype, seed=rows + K)
    check(fp4, orc, X, fmt, layout, "%s %s %s %s" % (fmt, dtype, layout, shape))


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_every_finite_bf16_value(fp4, orc, fmt):
    bits = np.arange(65536, dtype=np.uint32)
    finite = ((bits >> 7) & 0xFF) != 0xFF
    vals = bits[finite].astype(np.uint16)                     # 65280 patterns
    rng = np.random.default_rng(3)
    shuffled = rng.permutation(vals).reshape(255, 256)
    # sorted by magnitude: each block holds neighbouring values, so scales sit close to them
    by_mag = vals[np.argsort(vals & 0x7FFF, kind="stable")].reshape(255, 256)
    for layout in ("plain", "atom"):
        check(fp4, orc, shuffled, fmt, layout, "shuffled")
        check(fp4, orc, by_mag, fmt, layout, "by magnitude")


def tie_blocks(fmt, dtype):
    """Blocks whose largest magnitude fixes the scale exactly, filled with every E2M1
    midpoint times the scale and its neighbours one unit in the last place away."""
    vec = vec_of(fmt)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    if fmt == "nvfp4":
        sv = torch_scale_values("nvfp4")
        scales = [float(sv[c]) for c in range(1, 0x7F)]
        lead = 6.0
    else:
        scales = [2.0 ** k for k in range(-120, 121, 7)]
        lead = 4.0
    rows = []
    for s in scales:
        vals = np.concatenate([mids, -mids]) * s
        x32 = vals.astype(np.float32)
        if dtype == "bf16":
            u = x32.view(np.uint32) >> 16
            cand = np.concatenate([u, u + 1, u - 1]).astype(np.uint32) << 16
        else:
            u = x32.view(np.uint32)
            cand = np.concatenate([u, u + 1, u - 1]).astype(np.uint32)
        cand = cand.view(np.float32)
        for i in range(0, len(cand), vec - 1):
            blk = np.zeros(vec, np.float32)
            part = cand[i:i + vec - 1]
            blk[:len(part)] = part
            blk[-1] = np.float32(lead * s)
            rows.append(blk)
    while len(rows) % 4:
        rows.append(np.zeros(vec, np.float32))
    X = np.stack(rows).reshape(-1, vec * 4)
    return X if dtype == "f32" else W.to_bf16_bits(X)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_exact_ties_and_neighbours(fp4, orc, fmt, dtype):
    X = tie_blocks(fmt, dtype)
    for layout in ("plain", "atom"):
        check(fp4, orc, X, fmt, layout, "ties")


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_special_blocks(fp4, orc, fmt, dtype):
    vec = vec_of(fmt)
    blocks = [
        np.zeros(vec),                                   # zero block
        -np.zeros(vec),                                  # negative zeros
        np.full(vec, 2.0 ** -133),                       # bf16 subnormals
        np.linspace(-1e-38, 1e-38, vec),                 # fp32 subnormal range
        np.full(vec, 1e30), np.linspace(-3e38, 3e38, vec),   # saturating scales
        np.linspace(-6 * 448.0, 6 * 448.0, vec),          # largest unsaturated E4M3 scale
        np.r_[np.full(vec - 1, 1e-3), 1e3],              # one huge value: the rest round to 0
        np.r_[np.full(vec - 1, -1e-30), 5.0],            # tiny negatives -> code 8
        np.full(vec, 6 * 2.0 ** -10), np.full(vec, 6 * 2.0 ** -11),   # E4M3 zero / smallest scale edges
    ]
    X = np.stack([b.astype(np.float32) for b in blocks])
    X = np.repeat(X, 4, axis=0).reshape(-1, vec * 4)
    if dtype == "bf16":
        X = W.to_bf16_bits(X)
    for layout in ("plain", "atom"):
        check(fp4, orc, X, fmt, layout, "special")


@pytest.mark.parametrize("name", sorted(W.QUANT_WORKLOADS))
def test_named_workloads_full_size(fp4, orc, name):
    fmt, X = W.make_quant_workload(name)
    check(fp4, orc, X, fmt, "atom", name)


def test_plain_and_atom_agree_with_reorder(fp4):
    X = W.make_values(300, 2080, dtype="bf16", seed=9)
    for fmt in ("nvfp4", "mxfp4"):
        c1, plain = run_quant(fp4, X, fmt, "plain")
        c2, atom = run_quant(fp4, X, fmt, "atom")
        assert np.array_equal(c1, c2)
        vec = vec_of(fmt)
        pd = torch.from_numpy(plain).cuda()
        ad = torch.empty(fp4.scale_atom_bytes(300, 2080, vec), dtype=torch.uint8, device="cuda")
        fp4.scale_reorder(pd, ad, 300, 2080, vec)
        assert np.array_equal(ad.cpu().numpy(), atom)


def test_deterministic_and_stream_ordered(fp4):
    X = W.make_values(513, 1024, dtype="bf16", seed=10)
    s = torch.cuda.Stream()
    a = run_quant(fp4, X, "nvfp4", "atom")
    with torch.cuda.stream(s):
        b = run_quant(fp4, X, "nvfp4", "atom", stream=s)
    s.synchronize()
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_quantised_activations_feed_the_gemm(fp4, orc, fmt):
    """Device quantisation (atom scales) -> prepacked GEMM, against the oracle GEMM on
    the oracle's quantisation of the same values."""
    M, N, K = 200, 192, 1024
    vec = vec_of(fmt)
    Xa = W.make_values(M, K, dtype="bf16", seed=11)
    Xb = W.make_values(N, K, std=0.02, dtype="bf16", seed=12)
    devs = []
    for X, rows in ((Xa, M), (Xb, N)):
        Xd = torch.from_numpy(X.view(np.int16)).cuda()
        codes = torch.empty(rows * K // 2, dtype=torch.uint8, device="cuda")
        atoms = torch.empty(fp4.scale_atom_bytes(rows, K, vec), dtype=torch.uint8, device="cuda")
        fp4.quantize(fmt, Xd, rows, K, codes, atoms, in_dtype="bf16", layout="atom")
        devs += [codes, atoms]
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fp4.gemm(fmt, devs[0], devs[1], devs[2], devs[3], 1.0, D, M, N, K, "bf16", prepacked=True)
    assert fp4.get_device_status() == fp4.FP4_OK
    got = D.view(torch.int16).cpu().numpy().view(np.uint16)
    A, sfA = orc.quantize(Xa, fmt)
    B, sfB = orc.quantize(Xb, fmt)
    inp = W.GemmInputs(fmt, M, N, K, A, sfA, B, sfB, 1.0, "bf16", "quantised")
    ref, _ = orc.gemm_rows(inp)
    refb = orc.round_bf16(ref)
    err = np.abs(bf16_bits_to_f64(got) - bf16_bits_to_f64(refb))
    assert np.all(err <= bf16_ulp(refb))
