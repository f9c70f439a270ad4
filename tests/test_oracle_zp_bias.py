"""Pins of the oracle's zero-point and bias extension (weights stand for (w - zp) * scale; bias added to the sum).

None of the expected values comes from the function under test:
  - with no zero point and no bias it must reproduce the plain steps 1-11 exactly;
  - an integer zero point c is the same as shifting the integer weights to w - c (the integer matmuls are linear),
    so the result must equal the plain oracle on the shifted weights, exactly;
  - a bias adds itself, exactly, after the sum;
  - fractional zero points: the result stays within the closed-form MSD bound of the plain dequantized matmul
    x . ((w - zp) * scale) + bias, computed by an independent direct routine.
"""
import numpy as np
import pytest

import oracle
from weight_quantized_matmul_gb300 import inputs as I

MODES = (oracle.MODE_D, oracle.MODE_F)
HALF_C3 = 0.5 / (7.49 * 14.98 * 14.98)


@pytest.fixture(scope="module")
def oracle_mod():
    return oracle


def _zp_case(seed, M=6, K=512, N=72, G=64):
    """Weights in [-5, 4] and integer zero points in [-3, 3], so that w - zp stays an int4 value."""
    rng = np.random.default_rng(seed)
    wl = I.small_case(M, K, N, G, seed)
    x, _, sc = I.make_inputs(wl)
    w = rng.integers(-5, 5, size=(K, N)).astype(np.int8)
    zp = rng.integers(-3, 4, size=(K // G, N)).astype(np.float16)
    return x, w, zp, sc, G


@pytest.mark.parametrize("mode", MODES)
def test_no_zero_point_no_bias_is_the_plain_method(oracle_mod, mode):
    wl = I.small_case(5, 384, 80, 128, 21)
    x, wp, sc = I.make_inputs(wl)
    np.testing.assert_array_equal(oracle_mod.msd_matmul_ex(x, wp, sc, wl.G, mode=mode),
                                  oracle_mod.msd_matmul(x, wp, sc, wl.G, mode=mode))
    np.testing.assert_array_equal(oracle_mod.direct_matmul_ex(x, wp, sc, wl.G),
                                  oracle_mod.direct_matmul(x, wp, sc, wl.G))


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("seed", [1, 2])
def test_integer_zero_point_equals_shifted_weights(oracle_mod, mode, seed):
    x, w, zp, sc, G = _zp_case(seed)
    K, N = w.shape
    shifted = w - np.repeat(zp.astype(np.int8), G, axis=0)
    assert shifted.min() >= -8 and shifted.max() <= 7
    got = oracle_mod.msd_matmul_ex(x, I.pack_int4_along_k(w), sc, G, zero_point=zp, mode=mode)
    ref = oracle_mod.msd_matmul(x, I.pack_int4_along_k(shifted), sc, G, mode=mode)
    np.testing.assert_array_equal(got, ref)


def test_bias_adds_itself(oracle_mod):
    wl = I.small_case(4, 256, 64, 32, 23)
    x, wp, sc = I.make_inputs(wl)
    bias = np.linspace(-3.0, 5.0, wl.N).astype(np.float16)
    zp = np.full((wl.K // wl.G, wl.N), 0.5, dtype=np.float16)
    without = oracle_mod.msd_matmul_ex(x, wp, sc, wl.G, zero_point=zp)
    with_b = oracle_mod.msd_matmul_ex(x, wp, sc, wl.G, zero_point=zp, bias=bias)
    np.testing.assert_array_equal(with_b, without + bias.astype(np.float64)[None, :])
    d0 = oracle_mod.direct_matmul_ex(x, wp, sc, wl.G, zero_point=zp)
    d1 = oracle_mod.direct_matmul_ex(x, wp, sc, wl.G, zero_point=zp, bias=bias)
    np.testing.assert_array_equal(d1, d0 + bias.astype(np.float64)[None, :])


@pytest.mark.parametrize("G", [32, 128])
def test_fractional_zero_point_within_bound_of_direct_matmul(oracle_mod, G):
    wl = I.small_case(8, 512, 96, G, 29, x_dist="t3_clip60", scale_lo=-2.0, scale_hi=2.0)
    x, wp, sc = I.make_inputs(wl)
    rng = np.random.default_rng(31)
    zp = rng.uniform(-4.0, 4.0, size=(wl.K // G, wl.N)).astype(np.float16)
    bias = rng.uniform(-1.0, 1.0, size=wl.N).astype(np.float16)
    w = oracle_mod.decode_int4(wp, wl.K, wl.N).astype(np.float64)
    wz = np.abs(w - np.repeat(zp.astype(np.float64), G, axis=0))
    Gn = wl.K // G
    amax = np.abs(x.astype(np.float64)).reshape(wl.M, Gn, G).max(axis=2)
    bound = HALF_C3 * amax @ (np.abs(sc.astype(np.float64)) * wz.reshape(Gn, G, -1).sum(axis=1))
    yd = oracle_mod.direct_matmul_ex(x, wp, sc, G, zero_point=zp, bias=bias)
    y = oracle_mod.msd_matmul_ex(x, wp, sc, G, zero_point=zp, bias=bias)
    assert (np.abs(y - yd) <= bound + 1e-12 * np.abs(yd).max()).all()
    assert np.abs(y - yd).max() > 0.05 * bound.max()          # the bound is not vacuous
    # and the zero points matter: dropping them moves the result well outside the bound
    y0 = oracle_mod.msd_matmul_ex(x, wp, sc, G, bias=bias)
    assert np.abs(y0 - yd).max() > 10 * bound.max()
