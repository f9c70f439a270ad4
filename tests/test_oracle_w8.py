"""Pins of the oracle's int8-weight (W8) functions.

None of the expected values comes from the function under test:
  - with weights in the int4 range the W8 function must reproduce the (pinned) int4 path exactly;
  - a hand-worked one-row, two-k problem with weights at both ends of the int8 range;
  - the integer products are linear in the weights, so splitting w = 16 hi + lo (hi in [-8, 7], lo in [0, 15])
    must give 16 x the result on hi plus the result on lo (lo as an int4 value lo - 8 with zero point -8);
  - the result stays within the closed-form MSD bound of the plain dequantized matmul, itself checked against a
    numpy matrix product.
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


def _w8(seed, K, N, lo=-128, hi=127):
    return I.int_uniform(seed, 99, K * N, lo, hi).astype(np.int8).reshape(K, N)


@pytest.mark.parametrize("mode", MODES)
def test_w8_in_int4_range_is_the_int4_path(oracle_mod, mode):
    wl = I.small_case(5, 256, 40, 64, 31, w_dist="u7")
    x, _, sc = I.make_inputs(wl)
    w = I.make_w_int(wl)
    zp, bias = I.make_zero_point(wl, "frac"), I.make_bias(wl)
    got = oracle_mod.msd_matmul_w8(x, w, sc, wl.G, zero_point=zp, bias=bias, mode=mode)
    ref = oracle_mod.msd_matmul_ex(x, I.pack_int4_along_k(w), sc, wl.G, zero_point=zp, bias=bias, mode=mode)
    np.testing.assert_array_equal(got, ref)


def test_w8_hand_worked(oracle_mod):
    # x = [1, 0.5], one group of 2: A_max = 1; planes of 1: (7, 7, 5); of 0.5: t1 = 3.745 -> 4,
    # t2 = (3.745 - 4) 14.98 = -3.8199 -> -4, t3 = (-3.8199 + 4) 14.98 = 2.698 -> 3.
    # w = [100, -128]: Y1 = 700 - 512 = 188, Y2 = 700 + 512 = 1212, Y3 = 500 - 384 = 116.
    x = np.array([[1.0, 0.5]], dtype=np.float16)
    w = np.array([[100], [-128]], dtype=np.int8)
    sc = np.array([[1.0]], dtype=np.float16)
    want = 188 / 7.49 + 1212 / (7.49 * 14.98) + 116 / (7.49 * 14.98 * 14.98)
    got = oracle_mod.msd_matmul_w8(x, w, sc, 2, mode=oracle.MODE_D)
    assert abs(got[0, 0] - want) < 1e-12
    assert abs(oracle_mod.direct_matmul_w8(x, w, sc, 2)[0, 0] - 36.0) < 1e-12


@pytest.mark.parametrize("mode", MODES)
def test_w8_is_sixteen_hi_plus_lo(oracle_mod, mode):
    wl = I.small_case(4, 384, 24, 128, 32)
    x, _, sc = I.make_inputs(wl)
    w = _w8(5, wl.K, wl.N)
    hi = (w.astype(np.int16) >> 4).astype(np.int8)                 # [-8, 7]
    lo = (w.astype(np.int16) & 15).astype(np.int8)                 # [0, 15]
    assert np.array_equal(16 * hi.astype(np.int16) + lo, w.astype(np.int16))
    got = oracle_mod.msd_matmul_w8(x, w, sc, wl.G, mode=mode)
    sc16 = (sc.astype(np.float64) * 16).astype(np.float16)         # exact: a power of two
    part_hi = oracle_mod.msd_matmul_ex(x, I.pack_int4_along_k(hi), sc16, wl.G, mode=mode)
    zp_lo = np.full(sc.shape, -8.0, dtype=np.float16)
    part_lo = oracle_mod.msd_matmul_ex(x, I.pack_int4_along_k(lo - 8), sc, wl.G, zero_point=zp_lo, mode=mode)
    np.testing.assert_allclose(got, part_hi + part_lo, rtol=1e-12, atol=1e-12 * np.abs(got).max())


def test_w8_direct_is_a_matrix_product(oracle_mod):
    wl = I.small_case(3, 128, 16, 32, 33)
    x, _, sc = I.make_inputs(wl)
    w = _w8(6, wl.K, wl.N)
    zp, bias = I.make_zero_point(wl, "int"), I.make_bias(wl)
    deq = (w.astype(np.float64) - np.repeat(zp.astype(np.float64), wl.G, axis=0)) * \
        np.repeat(sc.astype(np.float64), wl.G, axis=0)
    ref = x.astype(np.float64) @ deq + bias.astype(np.float64)
    np.testing.assert_allclose(oracle_mod.direct_matmul_w8(x, w, sc, wl.G, zero_point=zp, bias=bias), ref,
                               rtol=1e-12, atol=1e-9)


@pytest.mark.parametrize("mode", MODES)
def test_w8_within_closed_form_bound(oracle_mod, mode):
    wl = I.small_case(6, 512, 48, 128, 34, x_dist="t3_clip60")
    x, _, sc = I.make_inputs(wl)
    w = _w8(7, wl.K, wl.N)
    zp = I.make_zero_point(wl, "frac")
    got = oracle_mod.msd_matmul_w8(x, w, sc, wl.G, zero_point=zp, mode=mode)
    ref = oracle_mod.direct_matmul_w8(x, w, sc, wl.G, zero_point=zp)
    G, Gn = wl.G, wl.groups
    amax = np.abs(x.astype(np.float64)).reshape(wl.M, Gn, G).max(axis=2)           # [M, Gn]
    wz = np.abs(w.astype(np.float64).reshape(Gn, G, wl.N) - zp.astype(np.float64)[:, None, :]).sum(axis=1)
    bound = HALF_C3 * (amax[:, :, None] * wz[None] * np.abs(sc.astype(np.float64))[None]).sum(axis=1)
    # binary32 unfold: a few ulps of slack on top of the binary64 bound
    assert np.all(np.abs(got - ref) <= bound * (1 + 1e-6) + 1e-9)
