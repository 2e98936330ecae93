"""Pins for the CPU oracle (oracle/oracle.c). CPU only.

Each function of the oracle is pinned to something other than itself:

* decoders -- E2M1 against the OCP value table (tests/golden/e2m1_values.txt);
  E4M3 and E8M0 exhaustively against torch's float8_e4m3fn / float8_e8m0fnu
  casts (a library routine);
* the GEMM -- hand-worked examples (tests/golden/worked_examples.txt), closed
  forms (all-ones -> alpha*K; one-hot rows select one product), the exhaustive
  16x16 code-pair product table, exact rational brute force on small random
  problems, and metamorphic relations (scale doubling, absolute values);
* bf16 rounding -- hand-derived ties, the double-rounding trap, overflow and
  subnormals, and torch's float32 -> bfloat16 cast on float32-exact inputs;
* the scale reorder -- bijectivity onto the padded buffer, zero padding and
  block locality. Whether this byte layout is the one the tensor core reads
  is pinned only on the GPU, by GEMM parity.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import pytest

from tests._helpers import (e2m1_golden, exact_gemm, parse_worked_examples, torch_scale_values,
                            unpack_codes)
from workloads import GemmInputs, pack_codes


def _inp(fmt, A, sfA, B, sfB, M, N, K, alpha=1.0):
    return GemmInputs(fmt, M, N, K, np.asarray(A, np.uint8), np.asarray(sfA, np.uint8),
                      np.asarray(B, np.uint8), np.asarray(sfB, np.uint8), alpha, "f32")


ONE_SCALE = {"nvfp4": 0x38, "mxfp4": 127}   # E4M3 1.0 and E8M0 2^0


# ---- decoders -----------------------------------------------------------------

def test_e2m1_matches_ocp_table(oracle_mod):
    table = e2m1_golden()
    for c in range(16):
        v = oracle_mod.e2m1(c)
        assert v == table[c]
        assert math.copysign(1.0, v) == math.copysign(1.0, table[c])


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_scale_decode_matches_torch(oracle_mod, fmt):
    ref = torch_scale_values(fmt)
    dec = oracle_mod.e4m3 if fmt == "nvfp4" else oracle_mod.e8m0
    for c in range(256):
        v = dec(c)
        if math.isnan(ref[c]):
            assert math.isnan(v), c
        else:
            assert v == ref[c], (c, v, ref[c])


def test_e4m3_landmarks(oracle_mod):
    # largest finite, smallest normal, smallest subnormal, and the two NaNs
    assert oracle_mod.e4m3(0x7E) == 448.0
    assert oracle_mod.e4m3(0x08) == 2.0 ** -6
    assert oracle_mod.e4m3(0x01) == 2.0 ** -9
    assert math.isnan(oracle_mod.e4m3(0x7F)) and math.isnan(oracle_mod.e4m3(0xFF))
    assert oracle_mod.e8m0(0) == 2.0 ** -127 and oracle_mod.e8m0(254) == 2.0 ** 127


# ---- the GEMM ------------------------------------------------------------------

def test_worked_examples(oracle_mod):
    for inp, D in parse_worked_examples():
        got, _ = oracle_mod.gemm_rows(inp)
        np.testing.assert_array_equal(got, D, err_msg=inp.name)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("K", [32, 64, 96, 256, 1056])
def test_all_ones_gives_alpha_K(oracle_mod, fmt, K):
    M, N = 3, 5
    vec = 16 if fmt == "nvfp4" else 32
    A = np.full((M, K // 2), 0x22, np.uint8)           # every code 2 = 1.0
    B = np.full((N, K // 2), 0x22, np.uint8)
    sfA = np.full((M, K // vec), ONE_SCALE[fmt], np.uint8)
    sfB = np.full((N, K // vec), ONE_SCALE[fmt], np.uint8)
    D, absd = oracle_mod.gemm_rows(_inp(fmt, A, sfA, B, sfB, M, N, K, alpha=0.75))
    assert np.all(D == 0.75 * K) and np.all(absd == 0.75 * K)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_one_hot_selects_single_product(oracle_mod, fmt):
    rng = np.random.default_rng(7)
    table = e2m1_golden()
    sv = torch_scale_values(fmt)
    vec = 16 if fmt == "nvfp4" else 32
    M, N, K = 6, 7, 192
    ka = rng.integers(0, K, M)
    kb = rng.integers(0, K, N)
    kb[:3] = ka[:3]                                  # force some matches
    ca = rng.integers(1, 16, M)
    cb = rng.integers(1, 16, N)
    ca[ca == 8] = 9
    cb[cb == 8] = 9
    codes_a = np.zeros((M, K), np.uint8)
    codes_b = np.zeros((N, K), np.uint8)
    codes_a[np.arange(M), ka] = ca
    codes_b[np.arange(N), kb] = cb
    lo, hi = (0x20, 0x58) if fmt == "nvfp4" else (120, 135)
    sfA = rng.integers(lo, hi, (M, K // vec)).astype(np.uint8)
    sfB = rng.integers(lo, hi, (N, K // vec)).astype(np.uint8)
    D, _ = oracle_mod.gemm_rows(_inp(fmt, pack_codes(codes_a), sfA, pack_codes(codes_b), sfB, M, N, K))
    for i in range(M):
        for j in range(N):
            if ka[i] == kb[j]:
                want = (table[ca[i]] * sv[sfA[i, ka[i] // vec]]) * (table[cb[j]] * sv[sfB[j, kb[j] // vec]])
            else:
                want = 0.0
            assert D[i, j] == want, (i, j)


def test_code_pair_products_exhaustive(oracle_mod):
    table = e2m1_golden()
    for fmt in ("nvfp4", "mxfp4"):
        vec = 16 if fmt == "nvfp4" else 32
        K = 64
        codes_a = np.zeros((16, K), np.uint8)
        codes_b = np.zeros((16, K), np.uint8)
        codes_a[:, 33] = np.arange(16)                  # odd k: high nibble
        codes_b[:, 33] = np.arange(16)
        sfA = np.full((16, K // vec), ONE_SCALE[fmt], np.uint8)
        sfB = np.full((16, K // vec), ONE_SCALE[fmt], np.uint8)
        D, _ = oracle_mod.gemm_rows(_inp(fmt, pack_codes(codes_a), sfA, pack_codes(codes_b), sfB, 16, 16, K))
        for a in range(16):
            for b in range(16):
                assert D[a, b] == table[a] * table[b], (fmt, a, b)


def _random_small(fmt, M, N, K, seed, wide_scales=False):
    rng = np.random.default_rng(seed)
    vec = 16 if fmt == "nvfp4" else 32
    A = rng.integers(0, 256, (M, K // 2)).astype(np.uint8)
    B = rng.integers(0, 256, (N, K // 2)).astype(np.uint8)
    if fmt == "nvfp4":
        hi = 0x7F if wide_scales else 0x60                # 0x7F is NaN: excluded
        sfA = rng.integers(0, hi, (M, K // vec)).astype(np.uint8)
        sfB = rng.integers(0, hi, (N, K // vec)).astype(np.uint8)
    else:
        lo, hi = (0, 255) if wide_scales else (120, 136)
        sfA = rng.integers(lo, hi, (M, K // vec)).astype(np.uint8)
        sfB = rng.integers(lo, hi, (N, K // vec)).astype(np.uint8)
    alpha = float(rng.choice([1.0, 0.5, -2.0, 1.0 / 3.0]))
    return _inp(fmt, A, sfA, B, sfB, M, N, K, alpha)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("seed", range(6))
def test_brute_force_exact_rational(oracle_mod, fmt, seed):
    rng = np.random.default_rng(100 + seed)
    M, N = int(rng.integers(1, 4)), int(rng.integers(1, 4))
    K = int(rng.choice([32, 64, 96, 160]))
    wide = seed % 2 == 1
    inp = _random_small(fmt, M, N, K, seed, wide_scales=wide)
    D, absd = oracle_mod.gemm_rows(inp)
    exact, exact_abs = exact_gemm(inp)
    for i in range(M):
        for j in range(N):
            if wide:
                # scales over the whole format range: the fp64 sum may round; each
                # of the K additions and the alpha multiply err by <= 2^-53 relative
                bound = (K + 2) * 2.0 ** -53 * float(exact_abs[i][j])
                assert abs(D[i, j] - float(exact[i][j])) <= bound, (i, j)
            else:
                # narrow scales keep every partial sum exact in fp64: only the final
                # multiply by alpha rounds
                unscaled = exact[i][j] / Fraction(inp.alpha)
                assert Fraction(float(unscaled)) == unscaled
                assert D[i, j] == float(unscaled) * inp.alpha, (i, j)
            assert absd[i, j] == pytest.approx(float(exact_abs[i][j]), rel=(K + 2) * 2.0 ** -52)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_scale_doubling_doubles_one_block(oracle_mod, fmt):
    inp = _random_small(fmt, 4, 3, 128, 11)
    inp.alpha = 1.0                                   # narrow scales + alpha 1: every sum exact
    vec = inp.vec
    D0, _ = oracle_mod.gemm_rows(inp)
    # contribution of block (row 2 of A, block 1) alone: zero every other code of A's row 2
    codes = unpack_codes(inp.A, inp.K)
    only = codes.copy()
    only[2, :] = 0
    only[2, vec:2 * vec] = codes[2, vec:2 * vec]
    inp_only = _inp(fmt, pack_codes(only), inp.sfA, inp.B, inp.sfB, 4, 3, 128, inp.alpha)
    Donly, _ = oracle_mod.gemm_rows(inp_only)
    sfA2 = inp.sfA.copy()
    sfA2[2, 1] += 8 if fmt == "nvfp4" else 1          # exponent + 1 = value x2
    inp2 = _inp(fmt, inp.A, sfA2, inp.B, inp.sfB, 4, 3, 128, inp.alpha)
    D2, _ = oracle_mod.gemm_rows(inp2)
    np.testing.assert_array_equal(np.delete(D2, 2, 0), np.delete(D0, 2, 0))
    np.testing.assert_array_equal(D2[2] - D0[2], Donly[2])


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_absdot_is_sum_of_magnitudes(oracle_mod, fmt):
    inp = _random_small(fmt, 5, 4, 96, 3)
    D, absd = oracle_mod.gemm_rows(inp)
    # clearing every sign bit (codes and alpha) turns the signed sum into the absolute one
    A_abs = inp.A & 0x77
    B_abs = inp.B & 0x77
    mag = _inp(fmt, A_abs, inp.sfA, B_abs, inp.sfB, 5, 4, 96, abs(inp.alpha))
    Dm, _ = oracle_mod.gemm_rows(mag)
    np.testing.assert_allclose(absd, Dm, rtol=1e-14)
    assert np.all(np.abs(D) <= absd * (1 + 1e-12))


def test_rows_and_pairs_agree(oracle_mod):
    inp = _random_small("nvfp4", 9, 11, 256, 5)
    D, absd = oracle_mod.gemm_rows(inp)
    rows = np.array([8, 0, 3])
    Dr, _ = oracle_mod.gemm_rows(inp, rows)
    np.testing.assert_array_equal(Dr, D[rows])
    ii, jj = np.meshgrid(np.arange(9), np.arange(11), indexing="ij")
    Dp, ap = oracle_mod.gemm_pairs(inp, ii.ravel(), jj.ravel())
    np.testing.assert_array_equal(Dp.reshape(9, 11), D)
    np.testing.assert_array_equal(ap.reshape(9, 11), absd)


def test_transpose_symmetry(oracle_mod):
    # D(A, B)^T == D(B, A): catches a transposed operand or a swapped scale
    inp = _random_small("mxfp4", 4, 6, 128, 9)
    D, _ = oracle_mod.gemm_rows(inp)
    sw = _inp("mxfp4", inp.B, inp.sfB, inp.A, inp.sfA, 6, 4, 128, inp.alpha)
    Dt, _ = oracle_mod.gemm_rows(sw)
    np.testing.assert_array_equal(Dt, D.T)


def test_rejects_bad_arguments(oracle_mod):
    inp = _random_small("nvfp4", 2, 2, 64, 1)
    with pytest.raises(ValueError):
        oracle_mod.gemm_rows(inp, rows=[5])
    with pytest.raises(ValueError):
        oracle_mod.gemm_pairs(inp, [0], [2])


# ---- output rounding -----------------------------------------------------------

def test_bf16_rounding_cases(oracle_mod):
    r = lambda x: int(oracle_mod.round_bf16(np.array([x]))[0])
    assert r(1.0) == 0x3F80
    assert r(1.0 + 2 ** -8) == 0x3F80                    # tie -> even (down)
    assert r(1.0 + 3 * 2 ** -8) == 0x3F82                # tie -> even (up)
    assert r(1.0 + 2 ** -8 + 2 ** -30) == 0x3F81         # one rounding, not via fp32
    assert r(-2.0) == 0xC000
    assert r(0.0) == 0x0000 and r(-0.0) == 0x8000
    assert r(3.0e38) == 0x7F62 or r(3.0e38) == 0x7F61    # finite
    assert r(2.0 ** 128) == 0x7F80 and r(-(2.0 ** 128)) == 0xFF80
    assert r((2 - 2 ** -8) * 2 ** 127) == 0x7F80         # tie above max finite -> inf
    assert r((2 - 2 ** -7) * 2 ** 127) == 0x7F7F
    assert r(2.0 ** -133) == 0x0001                      # smallest subnormal
    assert r(2.0 ** -134) == 0x0000                      # tie -> even (zero)
    assert r(1.5 * 2.0 ** -134) == 0x0001
    assert r(2.0 ** -126) == 0x0080                      # smallest normal
    assert r(float('nan')) & 0x7FFF > 0x7F80                 # NaN stays NaN


def test_bf16_rounding_matches_torch_on_f32_values(oracle_mod):
    import torch
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-60, 60, 20000))).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle_mod.round_bf16(x.astype(np.float64))
    np.testing.assert_array_equal(got, want)


def test_f32_rounding(oracle_mod):
    assert oracle_mod.round_f32(1.0 + 2 ** -24) == 1.0
    assert oracle_mod.round_f32(1.0 + 3 * 2 ** -24) == 1.0 + 2 ** -22


# ---- scale reorder --------------------------------------------------------------

@pytest.mark.parametrize("rows,ksf", [(128, 4), (300, 18), (1, 2), (257, 9), (128, 256)])
def test_scale_reorder_bijective_and_padded(oracle_mod, rows, ksf):
    # tag every byte with a unique id so the permutation can be followed
    n = rows * ksf
    ids = np.arange(n, dtype=np.int64)
    nbytes = oracle_mod.scale_atom_bytes(rows, ksf)
    assert nbytes == ((rows + 127) // 128) * ((ksf + 3) // 4) * 512
    where = np.full(n, -1, np.int64)
    # the oracle moves bytes; run it 3 times on the base-256 digits of the ids
    digits = [(ids >> (8 * d)) & 0xFF for d in range(3)]
    outs = [oracle_mod.scale_reorder(dg.astype(np.uint8), rows, ksf).astype(np.int64) for dg in digits]
    marker = oracle_mod.scale_reorder(np.ones(n, np.uint8), rows, ksf)
    placed = np.nonzero(marker)[0]
    assert placed.size == n                                   # injective onto n slots
    assert np.all(np.delete(marker, placed) == 0)             # padding stays zero
    got_ids = outs[0][placed] | (outs[1][placed] << 8) | (outs[2][placed] << 16)
    assert np.unique(got_ids).size == n
    where[got_ids] = placed
    r = ids // ksf
    c = ids % ksf
    atom = where // 512
    # block locality: a 512-byte atom holds exactly one 128-row x 4-column block,
    # atoms run along K first (ceil(ksf/4) per 128-row block)
    kc4 = (ksf + 3) // 4
    assert np.all(atom == (r // 128) * kc4 + c // 4)
    # inside an atom, each 16-byte line holds 4 rows 32 apart, 4 columns each
    line = (where % 512) // 16
    assert np.all(line == r % 32)


def test_scale_reorder_small_by_hand(oracle_mod):
    # rows 0, 32, 64, 96 of one atom share line 0; row 1 starts line 1
    sf = np.zeros((128, 4), np.uint8)
    sf[0] = [1, 2, 3, 4]
    sf[32] = [5, 6, 7, 8]
    sf[64, 0] = 9
    sf[96, 3] = 10
    sf[1, 0] = 11
    out = oracle_mod.scale_reorder(sf, 128, 4)
    assert list(out[0:16]) == [1, 2, 3, 4, 5, 6, 7, 8, 9, 0, 0, 0, 0, 0, 0, 10]
    assert out[16] == 11 and out.size == 512
