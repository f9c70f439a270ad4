"""The tight bar of the parity tests must see a wrong combine constant that the stated bar lets through.

A copy of the oracle with the third combine term (page section 4.1, step 10, Y3 / (7.49 * 14.98^2)) 10% too large
stands for a kernel with that mistake: its fp16-rounded output passes |y - y_ref| <= 2e-3 max|y_ref| + 1 ulp but
fails the tight bar, while the correct oracle's own fp16-rounded output passes both. The mistake is planted in a
copy of the oracle, on the CPU.
"""
import os

import numpy as np
import pytest

import oracle
import tolerance as T
from weight_quantized_matmul_gb300 import inputs as I

SRC = os.path.join(os.path.dirname(oracle.__file__), "wqbmm_oracle.c")

CASES = [I.small_case(4, 1024, 512, 128, seed=21), I.small_case(8, 4096, 256, 64, seed=22, x_dist="t3_clip60"),
         I.small_case(2, 2048, 384, 32, seed=23, x_dist="uniform3", w_dist="u7", scale_lo=-3.0, scale_hi=3.0)]


@pytest.fixture(scope="module")
def c3_too_large(tmp_path_factory):
    with open(SRC) as f:
        src = f.read()
    anchor = "y3 / (7.49 * 14.98 * 14.98)"
    assert anchor in src
    lib = oracle.build_variant(src.replace(anchor, "1.1 * " + anchor, 1), str(tmp_path_factory.mktemp("c3")),
                               "c3")
    return oracle.Oracle(lib)


@pytest.mark.parametrize("wl", CASES, ids=[c.name for c in CASES])
def test_tight_bar_sees_a_wrong_third_term(c3_too_large, wl):
    x, wp, sc = I.make_inputs(wl)
    ref_d = oracle.msd_matmul(x, wp, sc, wl.G, mode=oracle.MODE_D)
    ref_f = oracle.msd_matmul(x, wp, sc, wl.G, mode=oracle.MODE_F)
    good = ref_f.astype(np.float16)
    T.assert_matches(good, ref_d, ref_f, "correctly rounded")
    bad = c3_too_large.msd_matmul(x, wp, sc, wl.G, mode=oracle.MODE_F).astype(np.float16)
    T.assert_within_tolerance(bad, ref_d, "stated bar")           # the stated bar alone lets it through
    with pytest.raises(AssertionError):
        T.assert_tight(bad, ref_f, "planted")


def test_exact_rounding_sits_near_a_quarter_ulp():
    wl = I.small_case(16, 2048, 512, 128, seed=24)
    x, wp, sc = I.make_inputs(wl)
    ref_f = oracle.msd_matmul(x, wp, sc, wl.G, mode=oracle.MODE_F)
    e = T.tight_errors(ref_f.astype(np.float16), ref_f)
    assert e.max() <= 0.5 + 1e-9 and 0.2 <= e.mean() <= 0.3
