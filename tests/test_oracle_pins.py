"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Method: WeightQuantBatchMatmulExperiment page, section 4.1 (the eleven MSD steps), 4.2 (spec), 4.3 (int4 packing).
What pins what:
  - fp16 decode: every one of the 65536 bit patterns against numpy's own float16 conversion;
  - int4 decode: a hand-decoded fixture, and the round trip through the input generator's independent packer;
  - unfold: hand-worked values, the plane bound |A_i| <= 7, the telescoping reconstruction bound
    |x/A_max - (A1/7.49 + A2/(7.49*14.98) + A3/(7.49*14.98^2))| <= 0.5/(7.49*14.98^2), an exhaustive fp16 sweep;
  - steps 9-11: hand-worked 2x2 and 4x4 problems, the closed-form bound against the plain dequantized matmul,
    identity weights (the product returns x within the bound), all-ones weights (row sums of the planes), constant
    groups (R(1) times the column sums), zero groups, sign symmetry, and group / column permutation invariances.
"""
import numpy as np
import pytest

from golden_io import as_array, blocks, csv_rows
from weight_quantized_matmul_gb300 import inputs as I

C1 = 1.0 / 7.49
C2 = 1.0 / (7.49 * 14.98)
C3 = 1.0 / (7.49 * 14.98 * 14.98)
HALF_C3 = 0.5 * C3
MODES = (0, 1)   # binary64 unfold, binary32 unfold


def recon(planes):
    return planes[0] * C1 + planes[1] * C2 + planes[2] * C3


def rand_problem(M, K, N, G, seed, x_dist="normal", w_dist="u8", lo=0.005, hi=0.02, sigma=1.0):
    wl = I.small_case(M, K, N, G, seed, x_dist=x_dist, w_dist=w_dist, scale_lo=lo, scale_hi=hi, x_sigma=sigma)
    return I.make_inputs(wl)


# ---------------------------------------------------------------- decoding

def test_half_decode_all_bit_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_mod.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_int4_decode_hand_fixture(oracle_mod):
    b = blocks("int4_packing.txt")
    packed = as_array(b["packed"], np.uint8)
    want = as_array(b["weights"], np.int8)
    assert np.array_equal(oracle_mod.decode_int4(packed, 4, 3), want)


def test_int4_roundtrip_with_generator_packer(oracle_mod):
    w = I.int_uniform(11, 1, 64 * 48, -8, 7).astype(np.int8).reshape(64, 48)
    assert np.array_equal(oracle_mod.decode_int4(I.pack_int4_along_k(w), 64, 48), w)


# ---------------------------------------------------------------- unfold (steps 1-8)

def test_worked_unfold_values(oracle_mod):
    head, rows = csv_rows("unfold_worked_values.txt")
    assert head == ["x", "A1", "A2", "A3"]
    for r in rows:
        if r[0] == "R1":
            r1 = float(r[1])
            continue
        x = np.array([[1.0, float(r[0])]], dtype=np.float16)
        assert float(x[0, 1]) == float(r[0]), "fixture x must be exact in fp16"
        for mode in MODES:
            planes, amax = oracle_mod.unfold(x, 2, mode)
            assert amax[0, 0] == 1.0
            assert list(planes[:, 0, 1]) == [int(r[1]), int(r[2]), int(r[3])], (r, mode)
            assert list(planes[:, 0, 0]) == [7, 7, 5]
    assert recon(np.array([7, 7, 5])) == pytest.approx(r1, abs=1e-10)


def test_binary32_ties_round_half_even(oracle_mod):
    head, rows = csv_rows("unfold_ties_binary32.txt")
    for r in rows:
        amax, xv = float(r[0]), float(r[1])
        x = np.array([[amax, xv]], dtype=np.float16)
        assert float(x[0, 0]) == amax and float(x[0, 1]) == xv
        pf, _ = oracle_mod.unfold(x, 2, 1)
        pd, _ = oracle_mod.unfold(x, 2, 0)
        assert list(pf[:, 0, 1]) == [int(v) for v in r[2:5]]
        assert list(pd[:, 0, 1]) == [int(v) for v in r[5:8]]


@pytest.mark.parametrize("x_dist,sigma", [("normal", 1.0), ("t3_clip60", 1.0), ("normal_cols20", 1.0),
                                          ("uniform3", 3.0), ("normal", 1e-4)])
@pytest.mark.parametrize("G", [32, 64, 128])
def test_plane_bound_and_reconstruction(oracle_mod, x_dist, sigma, G):
    wl = I.small_case(24, 512, 16, G, 7, x_dist=x_dist, x_sigma=sigma)
    x = I.make_x(wl)
    xf = x.astype(np.float64)
    for mode in MODES:
        planes, amax = oracle_mod.unfold(x, G, mode)
        assert np.abs(planes).max() <= 7
        am = np.repeat(amax, G, axis=1)
        assert np.array_equal(am.reshape(24, -1, G).max(axis=2), np.abs(xf).reshape(24, -1, G).max(axis=2))
        err = np.abs(xf / am - recon(planes.astype(np.float64)))
        slack = 1e-12 if mode == 0 else 1e-6   # binary32 rounding of tmp1..tmp3 adds at most ~1e-7
        assert err.max() <= HALF_C3 + slack


def test_zero_group_gives_zero_planes(oracle_mod):
    x = np.zeros((2, 64), dtype=np.float16)
    x[1, 32:] = np.float16(0.75)
    for mode in MODES:
        planes, amax = oracle_mod.unfold(x, 32, mode)
        assert amax.tolist() == [[0.0, 0.0], [0.0, 0.75]]
        assert not planes[:, 0].any() and not planes[:, 1, :32].any()
        assert (planes[:, 1, 32:] == np.array([7, 7, 5])[:, None]).all()


def test_sign_symmetry_of_unfold(oracle_mod):
    x = I.make_x(I.small_case(8, 256, 16, 64, 3))
    for mode in MODES:
        p, a = oracle_mod.unfold(x, 64, mode)
        pn, an = oracle_mod.unfold(-x, 64, mode)
        assert np.array_equal(a, an) and np.array_equal(pn, -p)


@pytest.mark.parametrize("amax", [1.0, 3.0, 60.0, 0.0999755859375, 65504.0, 6.103515625e-05, 5.960464477539063e-08])
def test_exhaustive_fp16_sweep(oracle_mod, amax):
    """Every finite fp16 value v with |v| <= A_max, in a group [A_max, v] of size 2, through both precisions."""
    allv = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
    v = allv[np.isfinite(allv) & (np.abs(allv.astype(np.float64)) <= amax)]
    x = np.stack([np.full(v.shape, amax, dtype=np.float16), v], axis=1)
    vf = v.astype(np.float64)
    res = {}
    for mode in MODES:
        planes, am = oracle_mod.unfold(x, 2, mode)
        assert (am[:, 0] == float(np.float16(amax))).all()
        assert np.abs(planes).max() <= 7
        err = np.abs(vf / am[:, 0] - recon(planes[:, :, 1].astype(np.float64)))
        assert err.max() <= HALF_C3 + (1e-12 if mode == 0 else 1e-6)
        assert (planes[:, :, 0] == np.array([7, 7, 5])[:, None]).all()
        res[mode] = planes[:, :, 1]
    # the two precisions disagree only near rounding ties of tmp1..tmp3: rare
    differ = (res[0] != res[1]).any(axis=0).mean()
    assert differ < 2e-3


# ---------------------------------------------------------------- steps 9-11

def test_hand_2x2(oracle_mod):
    b = blocks("msd_hand_2x2.txt")
    x = as_array(b["x"], np.float16)
    w = as_array(b["w"], np.int8)
    sc = as_array(b["scale"], np.float16)
    wp = I.pack_int4_along_k(w)
    for mode in MODES:
        part = oracle_mod.group_partials(x, wp, 2, 2, 0, mode)
        for i, key in enumerate(("Y1", "Y2", "Y3")):
            assert np.array_equal(part[i], as_array(b[key], np.int32)), key
        y = oracle_mod.msd_matmul(x, wp, sc, 2, mode)
        np.testing.assert_allclose(y, as_array(b["y"], np.float64), rtol=0, atol=2e-10)
    np.testing.assert_array_equal(oracle_mod.direct_matmul(x, wp, sc, 2), as_array(b["y_direct"], np.float64))


def test_hand_4x4_two_groups(oracle_mod):
    b = blocks("msd_hand_4x4.txt")
    x = as_array(b["x"], np.float16)
    w = as_array(b["w"], np.int8)
    sc = as_array(b["scale (rows = groups)"], np.float16)
    wp = I.pack_int4_along_k(w)
    for mode in MODES:
        planes, amax = oracle_mod.unfold(x, 2, mode)
        np.testing.assert_array_equal(amax, as_array(b["amax"], np.float64))
        for i in range(3):
            np.testing.assert_array_equal(planes[i], as_array(b[f"planes A{i + 1}"], np.int8))
        for g in range(2):
            part = oracle_mod.group_partials(x, wp, 4, 2, g, mode)
            for i in range(3):
                np.testing.assert_array_equal(part[i], as_array(b[f"group {g} Y{i + 1}"], np.int32))
        # steps 10-11 from the hand partials
        want = np.zeros((4, 4))
        for g in range(2):
            yi = [as_array(b[f"group {g} Y{i + 1}"], np.float64) for i in range(3)]
            want += (yi[0] / 7.49 + yi[1] / (7.49 * 14.98) + yi[2] / (7.49 * 14.98 * 14.98)) \
                * amax[:, g:g + 1] * sc[g].astype(np.float64)[None, :]
        np.testing.assert_allclose(oracle_mod.msd_matmul(x, wp, sc, 2, mode), want, rtol=1e-13, atol=1e-13)


def msd_direct_bound(x, w_int, scale, G):
    """0.5/(7.49*14.98^2) * sum_g A_max[m,g] |scale[g,n]| sum_{k in g} |w[k,n]|."""
    M, K = x.shape
    Gn = K // G
    amax = np.abs(x.astype(np.float64)).reshape(M, Gn, G).max(axis=2)
    wabs = np.abs(w_int.astype(np.float64)).reshape(Gn, G, -1).sum(axis=1)
    return HALF_C3 * amax @ (np.abs(scale.astype(np.float64)) * wabs)


@pytest.mark.parametrize("x_dist,w_dist,G", [("normal", "u8", 128), ("t3_clip60", "u8", 64),
                                             ("normal_cols20", "pm1_mix", 32), ("uniform3", "u7", 128)])
def test_msd_within_closed_form_bound_of_direct_matmul(oracle_mod, x_dist, w_dist, G):
    wl = I.small_case(12, 512, 96, G, 5, x_dist=x_dist, w_dist=w_dist, scale_lo=-3.0, scale_hi=3.0)
    x, wp, sc = I.make_inputs(wl)
    w_int = oracle_mod.decode_int4(wp, wl.K, wl.N)
    bound = msd_direct_bound(x, w_int, sc, G)
    yd = oracle_mod.direct_matmul(x, wp, sc, G)
    for mode in MODES:
        y = oracle_mod.msd_matmul(x, wp, sc, G, mode)
        slack = 1e-12 * np.abs(yd).max() + (0 if mode == 0 else 1e-6 * bound.max() / HALF_C3)
        assert (np.abs(y - yd) <= bound + slack).all()
        # the bound is not vacuous: the error uses a real part of it
        assert np.abs(y - yd).max() > 0.05 * bound.max()


def test_identity_weights_return_x(oracle_mod):
    K = N = 256
    G = 128
    x = I.make_x(I.small_case(5, K, N, G, 9, x_dist="t3_clip60"))
    w = np.eye(K, dtype=np.int8)
    sc = np.ones((K // G, N), dtype=np.float16)
    amax = np.repeat(np.abs(x.astype(np.float64)).reshape(5, -1, G).max(axis=2), G, axis=1)
    for mode in MODES:
        y = oracle_mod.msd_matmul(x, I.pack_int4_along_k(w), sc, G, mode)
        assert (np.abs(y - x.astype(np.float64)) <= amax * (HALF_C3 + 1e-6)).all()


def test_all_ones_weights_give_plane_row_sums(oracle_mod):
    x = I.make_x(I.small_case(6, 256, 8, 64, 4))
    w = np.ones((256, 8), dtype=np.int8)
    wp = I.pack_int4_along_k(w)
    for mode in MODES:
        planes, _ = oracle_mod.unfold(x, 64, mode)
        for g in range(4):
            part = oracle_mod.group_partials(x, wp, 8, 64, g, mode)
            sums = planes[:, :, g * 64:(g + 1) * 64].astype(np.int32).sum(axis=2)
            assert np.array_equal(part, np.repeat(sums[:, :, None], 8, axis=2))


def test_constant_groups_scale_column_sums(oracle_mod):
    head, rows = csv_rows("unfold_worked_values.txt")
    r1 = float(rows[-1][1])
    M, K, N, G = 3, 256, 40, 64
    consts = np.array([[0.5, -2.0, 3.0, 0.125], [1.0, 1.0, -0.25, 7.5], [-60.0, 0.03125, 2.0, -1.5]])
    x = np.repeat(consts, G, axis=1).astype(np.float16)
    _, wp, sc = rand_problem(M, K, N, G, 13, lo=-2.0, hi=2.0)
    w = oracle_mod.decode_int4(wp, K, N).astype(np.float64)
    colsum = w.reshape(K // G, G, N).sum(axis=1)                       # [Gn, N]
    want = (consts * r1) @ (colsum * sc.astype(np.float64))
    for mode in MODES:
        # R(1) is stored to 10 significant digits
        np.testing.assert_allclose(oracle_mod.msd_matmul(x, wp, sc, G, mode), want, rtol=1e-9, atol=1e-9)


def test_zero_groups_contribute_nothing(oracle_mod):
    M, K, N, G = 4, 512, 32, 128
    x, wp, sc = rand_problem(M, K, N, G, 21)
    x[:, 128:256] = 0
    x[2, :] = 0
    w = oracle_mod.decode_int4(wp, K, N)
    w2 = w.copy()
    w2[128:256] = np.roll(w2[128:256], 1, axis=1)
    for mode in MODES:
        y = oracle_mod.msd_matmul(x, wp, sc, G, mode)
        assert np.array_equal(y, oracle_mod.msd_matmul(x, I.pack_int4_along_k(w2), sc, G, mode))
        assert not y[2].any()


def test_sign_and_scale_linearity(oracle_mod):
    M, K, N, G = 3, 256, 24, 64
    x, wp, sc = rand_problem(M, K, N, G, 17)
    for mode in MODES:
        y = oracle_mod.msd_matmul(x, wp, sc, G, mode)
        assert np.array_equal(oracle_mod.msd_matmul(-x, wp, sc, G, mode), -y)
        assert np.array_equal(oracle_mod.msd_matmul(x, wp, (sc.astype(np.float32) * 2).astype(np.float16), G, mode),
                              2 * y)


def test_group_and_column_permutation_invariance(oracle_mod):
    M, K, N, G = 4, 512, 48, 64
    x, wp, sc = rand_problem(M, K, N, G, 19, lo=-1.0, hi=1.0)
    w = oracle_mod.decode_int4(wp, K, N)
    gperm = np.array([5, 2, 7, 0, 3, 6, 1, 4])
    kperm = (gperm[:, None] * G + np.arange(G)[None, :]).reshape(-1)
    nperm = np.roll(np.arange(N), 7)[::-1]
    for mode in MODES:
        y = oracle_mod.msd_matmul(x, wp, sc, G, mode)
        yg = oracle_mod.msd_matmul(np.ascontiguousarray(x[:, kperm]), I.pack_int4_along_k(w[kperm]),
                                   np.ascontiguousarray(sc[gperm]), G, mode)
        np.testing.assert_allclose(yg, y, rtol=1e-12, atol=1e-12 * np.abs(y).max())
        yn = oracle_mod.msd_matmul(x, I.pack_int4_along_k(np.ascontiguousarray(w[:, nperm])),
                                   np.ascontiguousarray(sc[:, nperm]), G, mode)
        assert np.array_equal(yn, y[:, nperm])


def test_rows_argument_selects_rows(oracle_mod):
    M, K, N, G = 7, 256, 16, 128
    x, wp, sc = rand_problem(M, K, N, G, 23)
    full = oracle_mod.msd_matmul(x, wp, sc, G)
    rows = [6, 0, 3]
    assert np.array_equal(oracle_mod.msd_matmul(x, wp, sc, G, rows=rows), full[rows])
    part = oracle_mod.group_partials(x, wp, N, G, 1, rows=rows)
    assert np.array_equal(part, oracle_mod.group_partials(x, wp, N, G, 1)[:, rows])


def test_invalid_arguments_rejected(oracle_mod):
    x = np.zeros((2, 96), dtype=np.float16)
    with pytest.raises(ValueError):
        oracle_mod.unfold(x, 64)                  # K not a multiple of G
    with pytest.raises(ValueError):
        oracle_mod.msd_matmul(x, np.zeros((48, 8), np.uint8), np.zeros((3, 8), np.float16), 32, rows=[5])
