"""Pins for the oracle's fused epilogues (oracle_epilogue). CPU only.

* ReLU and squared ReLU: hand-worked values (negative, zero, negative zero,
  positive, with and without the bias);
* SwiGLU: silu checked against 50-digit arithmetic (mpmath, an independent
  implementation of exp) and the identity silu(-x) = silu(x) - x; the gate /
  up pairing on a hand example;
* the bias: added before the activation, column by column.
"""
from __future__ import annotations

import math

import numpy as np
import pytest


def test_relu_and_squared_relu_by_hand(oracle_mod):
    y = np.array([[-2.0, -0.0, 0.0, 0.5, 3.0]])
    assert oracle_mod.epilogue(y, None, "none").tolist() == y.tolist()
    assert oracle_mod.epilogue(y, None, "relu").tolist() == [[0.0, 0.0, 0.0, 0.5, 3.0]]
    assert oracle_mod.epilogue(y, None, "relu2").tolist() == [[0.0, 0.0, 0.0, 0.25, 9.0]]
    b = np.array([3.0, 1.0, -1.0, 0.25, -4.0], np.float32)
    # z = y + b = [1, 1, -1, 0.75, -1]
    assert oracle_mod.epilogue(y, b, "none").tolist() == [[1.0, 1.0, -1.0, 0.75, -1.0]]
    assert oracle_mod.epilogue(y, b, "relu").tolist() == [[1.0, 1.0, 0.0, 0.75, 0.0]]
    assert oracle_mod.epilogue(y, b, "relu2").tolist() == [[1.0, 1.0, 0.0, 0.5625, 0.0]]


def silu_50_digits(x: float) -> float:
    mpmath = pytest.importorskip("mpmath")
    with mpmath.workdps(50):
        v = mpmath.mpf(x)
        return float(v / (1 + mpmath.exp(-v)))


def test_swiglu_against_high_precision(oracle_mod):
    xs = np.concatenate([np.linspace(-30, 30, 241), [-1e-3, 1e-3, 0.0, 50.0, -50.0]])
    ups = np.linspace(-2, 2, xs.size)
    y = np.empty((1, 2 * xs.size))
    y[0, 0::2] = xs
    y[0, 1::2] = ups
    got = oracle_mod.epilogue(y, None, "swiglu")[0]
    want = np.array([silu_50_digits(x) * u for x, u in zip(xs, ups)])
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-300)


def test_silu_reflection_identity(oracle_mod):
    xs = np.linspace(-20, 20, 161)
    y = np.empty((2, 2 * xs.size))
    y[0, 0::2], y[1, 0::2] = xs, -xs
    y[:, 1::2] = 1.0
    out = oracle_mod.epilogue(y, None, "swiglu")
    assert np.all(np.abs(out[1] - (out[0] - xs)) <= 1e-12 * np.maximum(1.0, np.abs(xs)))


def test_swiglu_pairs_gate_then_up(oracle_mod):
    # gate = even column, up = odd column, bias added first
    y = np.array([[0.0, 5.0, 2.0, 3.0], [-1.0, 0.5, 1.0, -2.0]])
    b = np.array([1.0, -1.0, 0.0, 1.0], np.float32)
    got = oracle_mod.epilogue(y, b, "swiglu")
    s = lambda x: x / (1.0 + math.exp(-x))
    want = [[s(1.0) * 4.0, s(2.0) * 4.0], [s(0.0) * -0.5, s(1.0) * -1.0]]
    np.testing.assert_allclose(got, want, rtol=1e-15)
    assert got.shape == (2, 2)


def test_rejects_bad_arguments(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.epilogue(np.zeros((1, 3)), None, "swiglu")
