"""The seeded input generator: encoders, scale rules, packing, determinism. CPU only."""
from __future__ import annotations

import numpy as np
import pytest

import workloads as W
from tests._helpers import e2m1_golden, torch_scale_values, unpack_codes


def _decode_e2m1(codes):
    t = e2m1_golden()
    return np.vectorize(lambda c: t[int(c)])(codes)


def test_e2m1_encode_exact_grid_and_ties():
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c, v in enumerate(grid):
        assert W.encode_e2m1(np.array([v]))[0] == c
        assert W.encode_e2m1(np.array([-v]))[0] == c | 8
    # ties go to the even code
    ties = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for x, c in ties.items():
        assert W.encode_e2m1(np.array([x]))[0] == c, x
        assert W.encode_e2m1(np.array([-x]))[0] == c | 8, x
    # saturation
    assert W.encode_e2m1(np.array([7.9, 1e9]))[0] == 7
    assert W.encode_e2m1(np.array([-100.0]))[0] == 15


def test_e2m1_encode_is_nearest():
    rng = np.random.default_rng(0)
    x = rng.uniform(-7, 7, 20000)
    codes = W.encode_e2m1(x)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    dec = _decode_e2m1(codes)
    best = np.min(np.abs(np.abs(x)[:, None] - grid[None, :]), axis=1)
    assert np.all(np.abs(np.abs(dec) - np.minimum(np.abs(x), 6.0)) <= best + 1e-12)


def test_pack_low_nibble_first():
    codes = np.array([[1, 2, 3, 4]], np.uint8)
    assert list(W.pack_codes(codes)[0]) == [0x21, 0x43]
    np.testing.assert_array_equal(unpack_codes(W.pack_codes(codes), 4), codes)


def test_nvfp4_scale_rule():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((8, 64)).astype(np.float32)
    x[3, :16] = 0.0                                         # an all-zero block
    packed, sf = W.quantize_nvfp4(x)
    sv = torch_scale_values("nvfp4")
    amax = np.abs(x.reshape(8, 4, 16)).max(axis=2)
    for r in range(8):
        for b in range(4):
            s = sv[sf[r, b]]
            # the chosen byte is the E4M3 value nearest absmax/6
            cand = sv[:0x7F]
            assert abs(s - amax[r, b] / 6) <= np.min(np.abs(cand - amax[r, b] / 6)) + 1e-12
    assert np.all(unpack_codes(packed, 64)[3, :16] == 0) and sf[3, 0] == 0
    # codes are the nearest grid point of x / decoded scale
    codes = unpack_codes(packed, 64)
    dec = _decode_e2m1(codes) * np.repeat(sv[sf], 16, axis=1)
    err = np.abs(dec - x)
    assert np.all(err <= np.repeat(sv[sf], 16, axis=1) * 1.0 + 1e-6)


def test_mxfp4_scale_rule():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((4, 128)).astype(np.float32) * 3
    x[1, 32:64] = 0.0
    packed, sf = W.quantize_mxfp4(x)
    amax = np.abs(x.reshape(4, 4, 32)).max(axis=2)
    for r in range(4):
        for b in range(4):
            if amax[r, b] == 0:
                assert sf[r, b] == 0
            else:
                assert int(sf[r, b]) - 127 == int(np.floor(np.log2(amax[r, b]))) - 2
    codes = unpack_codes(packed, 128)
    assert np.all(codes[1, 32:64] == 0)
    # the largest element of every block lands on magnitude 4 or 6 (x/scale in [4, 8))
    mags = np.abs(_decode_e2m1(codes)).reshape(4, 4, 32).max(axis=2)
    assert np.all((mags == 4) | (mags == 6) | (amax == 0))


def test_uniform_codes_recipe():
    inp = W.make_config("nvfp4_128x128x256_f32")
    assert inp.A.shape == (128, 128) and inp.sfA.shape == (128, 16)
    codes = unpack_codes(inp.A, 256)
    assert set(np.unique(codes)) == set(range(16))
    sv = torch_scale_values("nvfp4")
    assert set(np.unique(sv[inp.sfA])) == {2.0 ** u for u in range(-3, 4)}


def test_generator_is_deterministic():
    a = W.make_random("nvfp4", 40, 30, 64, seed=5)
    b = W.make_random("nvfp4", 40, 30, 64, seed=5)
    c = W.make_random("nvfp4", 40, 30, 64, seed=6)
    for f in ("A", "sfA", "B", "sfB"):
        np.testing.assert_array_equal(getattr(a, f), getattr(b, f))
    assert not np.array_equal(a.A, c.A)


@pytest.mark.parametrize("name", W.config_names())
def test_config_shapes(name):
    s = W.config_shape(name)
    assert s["K"] % 32 == 0 and s["M"] > 0 and s["N"] > 0


def test_small_config_draw():
    inp = W.make_random("mxfp4", 17, 9, 96, dist="t3")
    assert inp.A.shape == (17, 48) and inp.sfA.shape == (17, 3)
