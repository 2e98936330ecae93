"""Pins for the oracle's grouped (mixture-of-experts) GEMM, grouped_gemm_rows. CPU only.

* a closed form: every A value 1 and every value of B_g equal to 2^g, so each
  D row is K * 2^g(row) -- which fails if a row is given another group's
  weights, if a group boundary is off by one, or if empty groups shift the
  others;
* exact brute force (Python fractions, scale bytes decoded by torch) per
  group on a small random problem, the groups sliced here from the
  definition: group g = rows offsets[g] .. offsets[g+1]-1 of A, rows
  g*N .. g*N+N-1 of B;
* a sampled subset of rows in shuffled order equals the same rows of the
  full result;
* planted mistakes (an off-by-one group boundary, the next group's weights)
  fail the closed form.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest

import workloads as W
from tests._helpers import exact_gemm

SIZES = [3, 0, 5, 1, 0, 2]      # empty groups included, one at the start of a run of rows


def _pack(codes):
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def closed_form_problem(fmt):
    N, K = 4, 64
    vec = 16 if fmt == "nvfp4" else 32
    offsets = np.concatenate([[0], np.cumsum(SIZES)]).astype(np.int64)
    M, G = int(offsets[-1]), len(SIZES)
    one = 2                                              # E2M1 code of 1.0
    A = _pack(np.full((M, K), one, np.uint8))
    B = _pack(np.full((G * N, K), one, np.uint8))
    if fmt == "nvfp4":                                   # E4M3 2^e: exponent field e + 7
        sfA = np.full((M, K // vec), 7 << 3, np.uint8)
        sfB = np.repeat(((np.arange(G) + 7) << 3).astype(np.uint8), N)[:, None].repeat(K // vec, 1)
    else:                                                # E8M0 2^e: byte e + 127
        sfA = np.full((M, K // vec), 127, np.uint8)
        sfB = np.repeat((np.arange(G) + 127).astype(np.uint8), N)[:, None].repeat(K // vec, 1)
    gin = W.GroupedInputs(fmt, offsets, N, K, A, sfA, np.ascontiguousarray(B), np.ascontiguousarray(sfB), 1.0, "f32")
    expect = np.array([K * 2.0 ** g for g, n in enumerate(SIZES) for _ in range(n)])
    return gin, expect


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_grouped_closed_form(oracle_mod, fmt):
    gin, expect = closed_form_problem(fmt)
    D, absd = oracle_mod.grouped_gemm_rows(gin)
    assert D.shape == (gin.M, gin.N)
    np.testing.assert_array_equal(D, expect[:, None].repeat(gin.N, 1))
    np.testing.assert_array_equal(absd, D)


def test_grouped_exact_brute_force(oracle_mod):
    sizes = [2, 0, 3, 1]
    gin = W.make_grouped("nvfp4", sizes, 3, 64, seed=4, alpha=0.5)
    D, absd = oracle_mod.grouped_gemm_rows(gin)
    K, N, ksf = gin.K, gin.N, gin.K // 16
    row = 0
    for g, m in enumerate(sizes):
        if m == 0:
            continue
        part = W.GemmInputs("nvfp4", m, N, K, gin.A[row:row + m], gin.sfA[row:row + m],
                            gin.B[g * N:(g + 1) * N], gin.sfB[g * N:(g + 1) * N], 0.5, "f32")
        ed, ea = exact_gemm(part)
        for i in range(m):
            for j in range(N):
                assert Fraction(D[row + i, j]) == ed[i][j]
                assert Fraction(absd[row + i, j]) == ea[i][j]
        row += m
    assert row == gin.M and ksf == gin.sfA.shape[1]


def test_grouped_sampled_rows(oracle_mod):
    gin = W.make_grouped("mxfp4", [40, 0, 130, 7], 24, 128, seed=2)
    full, fa = oracle_mod.grouped_gemm_rows(gin)
    rows = np.random.default_rng(0).permutation(gin.M)[:50]
    part, pa = oracle_mod.grouped_gemm_rows(gin, rows)
    np.testing.assert_array_equal(part, full[rows])
    np.testing.assert_array_equal(pa, fa[rows])


def test_grouped_pins_reject_off_by_one_boundary(oracle_mod, monkeypatch):
    monkeypatch.setattr(oracle_mod, "_group_of_rows",
                        lambda offsets, rows: np.searchsorted(offsets, rows, side="left") - 1)
    gin, expect = closed_form_problem("nvfp4")
    with pytest.raises(Exception):
        D, _ = oracle_mod.grouped_gemm_rows(gin)
        np.testing.assert_array_equal(D, expect[:, None].repeat(gin.N, 1))


def test_grouped_pins_reject_wrong_weights(oracle_mod, monkeypatch):
    real = oracle_mod._GroupProblem

    class NextGroupWeights(real):
        def __init__(self, gin, g):
            super().__init__(gin, g)
            n = int(gin.N)
            nxt = (g + 1) % gin.G
            self.B = gin.B.reshape(-1, gin.K // 2)[nxt * n:(nxt + 1) * n]
            self.sfB = gin.sfB.reshape(-1, gin.K // gin.vec)[nxt * n:(nxt + 1) * n]

    monkeypatch.setattr(oracle_mod, "_GroupProblem", NextGroupWeights)
    gin, expect = closed_form_problem("mxfp4")
    D, _ = oracle_mod.grouped_gemm_rows(gin)
    assert not np.array_equal(D, expect[:, None].repeat(gin.N, 1))
