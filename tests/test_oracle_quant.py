"""Pins for the oracle's quantisation step (oracle_quantize and its encoders). CPU only.

What pins each part, without comparing the oracle with itself:

* E2M1 encode -- exact rational brute force over the value table of
  tests/golden/e2m1_values.txt (nearest value, a tie goes to the even code),
  on every E2M1 midpoint, its fp32 neighbours, a fine grid and extremes;
* E4M3 encode -- the same brute force over torch's float8_e4m3fn decode of all
  non-negative finite bytes, and torch's own float32 -> float8_e4m3fn cast (a
  library routine, round to nearest even) below the saturation point;
* the quantiser -- round trips (values built from codes and a scale that the
  block's largest magnitude fixes come back as the same codes and scale),
  closed forms for the scale byte, zero blocks, the error bound of round to
  nearest on random data, and agreement with the input generator's quantiser
  (workloads/, numpy + torch), which was written separately from the same
  reading.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import pytest

from tests._helpers import e2m1_golden, torch_scale_values, unpack_codes


def f32(x) -> float:
    return float(np.float32(x))


def nearest_code(value: float, table: dict[int, float], codes) -> int:
    """Brute force: code whose value is nearest to `value` (exact rationals), tie -> even code."""
    v = Fraction(value)
    best = None
    for c in codes:
        d = abs(v - Fraction(table[c]))
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    return best[1]


def e2m1_expected(q: float) -> int:
    table = e2m1_golden()
    mag = nearest_code(abs(q), table, range(8))
    return mag | (8 if math.copysign(1.0, q) < 0 else 0)


def e2m1_probe_values() -> list[float]:
    table = e2m1_golden()
    mags = sorted({abs(table[c]) for c in range(8)})
    vals = [0.0, -0.0, 1e-45, -1e-45, 1e-30, -1e-30, 7.0, 7.999, 8.0, 100.0, 3e38, -3e38, -6.0, -6.5]
    for a, b in zip(mags, mags[1:]):
        mid = f32((a + b) / 2)
        for m in (mid, -mid):
            vals += [m, float(np.nextafter(np.float32(m), np.float32(np.inf))),
                     float(np.nextafter(np.float32(m), np.float32(-np.inf)))]
    for m in mags:
        vals += [m, -m]
    vals += [f32(k / 256.0) for k in range(-2048, 2049, 3)]
    return vals


def test_e2m1_encode_brute_force(oracle_mod):
    for q in e2m1_probe_values():
        assert oracle_mod.e2m1_encode(q) == e2m1_expected(q), q


def test_e2m1_encode_hand_cases(oracle_mod):
    # midpoint ties to the even code: 0.25->0, 0.75->1.0, 1.25->1.0, 1.75->2.0,
    # 2.5->2.0, 3.5->4.0, 5->4.0; saturation at 6; sign kept on zero
    cases = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6, 6.0: 7, 1e9: 7,
             0.26: 1, 2.51: 5, 5.01: 7, -0.0: 8, -0.2: 8, -0.3: 9, -7.0: 15}
    for q, c in cases.items():
        assert oracle_mod.e2m1_encode(q) == c, q


def e4m3_table() -> dict[int, float]:
    vals = torch_scale_values("nvfp4")
    return {c: float(vals[c]) for c in range(0x7F)}


def test_e4m3_encode_brute_force(oracle_mod):
    table = e4m3_table()
    probes = [0.0, 1e-45, 2.0 ** -10, 2.0 ** -11, 447.0, 448.0, 449.0, 464.0, 1e6, 3e38]
    ordered = sorted(table.values())
    for a, b in zip(ordered, ordered[1:]):
        mid = f32((a + b) / 2)
        assert mid == (a + b) / 2                      # midpoints are fp32-exact
        probes += [a, mid, float(np.nextafter(np.float32(mid), np.float32(0))),
                   float(np.nextafter(np.float32(mid), np.float32(np.inf)))]
    rng = np.random.default_rng(5)
    probes += [float(v) for v in rng.uniform(0, 460, 300).astype(np.float32)]
    probes += [float(v) for v in np.exp2(rng.uniform(-12, 9, 300)).astype(np.float32)]
    for v in probes:
        want = 0x7E if v >= 448.0 else nearest_code(v, table, range(0x7F))
        assert oracle_mod.e4m3_encode(v) == want, v


def test_e4m3_encode_matches_torch_cast(oracle_mod):
    import torch
    rng = np.random.default_rng(6)
    v = np.concatenate([rng.uniform(0, 448, 2000), np.exp2(rng.uniform(-12, 8.8, 2000))]).astype(np.float32)
    v = v[v <= 448]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle_mod.e4m3_encode(float(x)) for x in v], dtype=np.uint8)
    assert np.array_equal(got, ref)


# ---- the quantiser ------------------------------------------------------------------

def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 values that bf16 holds exactly -> their bf16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exact in bf16"
    return (u >> 16).astype(np.uint16)


def decode_codes(codes: np.ndarray, K: int) -> np.ndarray:
    table = e2m1_golden()
    lut = np.array([table[c] for c in range(16)], dtype=np.float64)
    return lut[unpack_codes(codes, K)]


def roundtrip_case(fmt, rows, K, seed):
    """Codes and scales whose blocks each hold a magnitude that fixes the scale."""
    vec = 16 if fmt == "nvfp4" else 32
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, size=(rows, K), dtype=np.uint8)
    nb = K // vec
    lead = rng.integers(0, vec, size=(rows, nb))
    if fmt == "nvfp4":
        # the block's largest magnitude is 6 s, so amax / 6 = s exactly
        big = rng.choice(np.array([7, 15], np.uint8), size=(rows, nb))
        sbytes = rng.integers(1, 0x7F, size=(rows, nb)).astype(np.uint8)
        svals = torch_scale_values("nvfp4")[sbytes]
    else:
        # 4 s <= amax < 8 s, so floor(log2 amax) - 2 = log2 s
        big = rng.choice(np.array([6, 7, 14, 15], np.uint8), size=(rows, nb))
        sbytes = rng.integers(2, 250, size=(rows, nb)).astype(np.uint8)
        svals = np.exp2(sbytes.astype(np.float64) - 127)
    for r in range(rows):
        for b in range(nb):
            codes[r, b * vec + lead[r, b]] = big[r, b]
    x = decode_codes(pack(codes), K) * np.repeat(svals, vec, axis=1)
    return codes, sbytes, x


def pack(codes: np.ndarray) -> np.ndarray:
    from workloads import pack_codes
    return pack_codes(codes)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_quantize_roundtrip(oracle_mod, fmt, dtype):
    rows, K = 6, 256
    codes, sbytes, x = roundtrip_case(fmt, rows, K, seed=11)
    x32 = x.astype(np.float32)
    assert np.array_equal(x32.astype(np.float64), x)              # exact in fp32
    X = x32 if dtype == "f32" else to_bf16_bits(x32)
    got_codes, got_sf = oracle_mod.quantize(X, fmt)
    assert np.array_equal(got_sf, sbytes)
    assert np.array_equal(unpack_codes(got_codes, K), codes)


def test_quantize_zero_blocks(oracle_mod):
    for fmt in ("nvfp4", "mxfp4"):
        x = np.zeros((2, 64), np.float32)
        x[1] = -0.0
        codes, sf = oracle_mod.quantize(x, fmt)
        assert np.all(sf == 0)
        c = unpack_codes(codes, 64)
        assert np.all(c[0] == 0)
        # NVFP4: a zero scale gives all-zero codes; MXFP4 keeps the sign of -0
        assert np.all(c[1] == (0 if fmt == "nvfp4" else 8))


def test_quantize_mx_scale_closed_form(oracle_mod):
    js = list(range(-140, 128, 3)) + [-127, -126, -125, -124, 126, 127]
    for j in js:
        top = np.float32(np.inf) if j + 1 >= 128 else np.float32(2.0 ** (j + 1))   # 2^128 is past fp32
        for amax in (2.0 ** j, float(np.nextafter(top, np.float32(0)))):
            if amax == 0 or not np.isfinite(np.float32(amax)):
                continue
            x = np.zeros((1, 32), np.float32)
            x[0, 5] = -amax
            _, sf = oracle_mod.quantize(x, "mxfp4")
            e = math.frexp(float(np.float32(amax)))[1] - 1      # floor(log2 amax)
            assert sf[0, 0] == min(max(e - 2, -127), 127) + 127, (j, amax)


def test_quantize_nv_scale_saturates(oracle_mod):
    x = np.zeros((1, 16), np.float32)
    for amax, code in ((6 * 448.0, 0x7E), (1e30, 0x7E), (6 * 2.0 ** -9, 0x01), (2.0 ** -11, 0x00)):
        x[0, 3] = amax
        _, sf = oracle_mod.quantize(x, "nvfp4")
        assert sf[0, 0] == code, amax


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_quantize_error_bound(oracle_mod, fmt):
    """Round to nearest: |x - x^| <= s * half the E2M1 spacing at x/s (saturated above 6)."""
    vec = 16 if fmt == "nvfp4" else 32
    rng = np.random.default_rng(12)
    x = (rng.standard_t(3, size=(64, 512)) * np.exp2(rng.integers(-16, 12, size=(64, 1)))).astype(np.float32)
    codes, sf = oracle_mod.quantize(x, fmt)
    svals = torch_scale_values(fmt)[sf]
    s = np.repeat(svals, vec, axis=1)
    xh = decode_codes(codes, 512) * s
    # an NVFP4 block whose amax / 6 rounds to a zero scale is all zeros
    zero = s == 0
    assert np.all(xh[zero] == 0) and np.all(np.abs(x[zero]) <= 6 * 2.0 ** -10)
    q = np.abs(x.astype(np.float64)) / np.where(zero, 1.0, s)
    half = np.where(q <= 2, 0.25, np.where(q <= 4, 0.5, 1.0))
    err = np.abs(x - xh)
    ok = np.where(q <= 6, err <= half * s * (1 + 2.0 ** -20), np.abs(xh) == 6 * s)
    assert ok[~zero].all()
    assert np.all((np.sign(xh) == np.sign(x)) | (xh == 0))
    # the scale brackets the block maximum: amax / s in (3, 6.5] (NVFP4 normal
    # scales, within half an E4M3 step of amax / 6) or [4, 8) (MXFP4)
    amax = np.abs(x.astype(np.float64)).reshape(64, -1, vec).max(axis=2)
    if fmt == "nvfp4":
        normal = (svals >= 2.0 ** -6) & (amax < 6 * 448.0)
        assert normal.sum() > 1000
        ratio = amax[normal] / svals[normal]
        assert np.all((ratio > 6 / (1 + 2.0 ** -4) - 1e-9) & (ratio < 6 / (1 - 2.0 ** -4) + 1e-9))
    else:
        ratio = amax / svals
        assert np.all((ratio >= 4) & (ratio < 8))


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_quantize_matches_input_generator(oracle_mod, fmt):
    from workloads import quantize_mxfp4, quantize_nvfp4
    rng = np.random.default_rng(13)
    x = rng.standard_normal((32, 256)).astype(np.float32)
    x[3, :16] = 0
    x[5, 40] = 1000.0
    want_codes, want_sf = (quantize_nvfp4 if fmt == "nvfp4" else quantize_mxfp4)(x)
    codes, sf = oracle_mod.quantize(x, fmt)
    assert np.array_equal(sf, want_sf)
    assert np.array_equal(codes, want_codes)


def test_quantize_bf16_input_widens_exactly(oracle_mod):
    rng = np.random.default_rng(14)
    x = rng.standard_normal((8, 64)).astype(np.float32)
    x = (x.view(np.uint32) & 0xFFFF0000).view(np.float32)     # bf16-exact values
    for fmt in ("nvfp4", "mxfp4"):
        a = oracle_mod.quantize(x, fmt)
        b = oracle_mod.quantize(to_bf16_bits(x), fmt)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_quantize_rejects_bad_arguments(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.quantize(np.zeros((2, 48), np.float32), "mxfp4")
