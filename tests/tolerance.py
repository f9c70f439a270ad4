"""Comparison bars of the GPU parity tests (method: WeightQuantBatchMatmulExperiment page, section 4.1).

Two bars for the fp16 output y of steps 1-11:

  within_tolerance  the stated bar, |y - y_ref| <= 2e-3 * max|y_ref| + 1 fp16 ulp(y_ref), element by element;

  tight             for the outputs that are not small (|y_ref| >= max|y_ref| / 16), where the binary32 arithmetic of
                    the combine and the accumulation is far below one fp16 ulp: the GPU result must be y_ref rounded
                    to fp16, up to 0.6 fp16 ulp(y_ref). y_ref is the oracle with the binary32 unfold (the GPU's planes
                    exactly), in binary64 from step 9 on. Rounding the exact value gives at most 0.5 ulp; the 0.1 ulp
                    left covers the binary32 rounding of the constants, of the three-term combine and of the sum
                    over the groups (relative size about 1e-6, a few thousandths of an ulp) with a wide margin. A
                    wrong combine constant shows here long before it shows against the stated bar: an error of 10% in
                    the third term moves typical outputs by 0.5 to 1 ulp. The mean error of those outputs must also
                    stay below 0.3 ulp (exact rounding gives about 0.25).
"""
import numpy as np

TIGHT_ULP = 0.6
TIGHT_MEAN_ULP = 0.3
TIGHT_FLOOR = 1.0 / 16


def fp16_ulp(v):
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -14)))
    return 2.0 ** (e - 10)


def assert_within_tolerance(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    tol = 2e-3 * np.abs(ref).max() + fp16_ulp(ref)
    err = np.abs(got - ref)
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())}/{bad.size} outside tolerance, max err {err.max():.4g}, "
                           f"max |ref| {np.abs(ref).max():.4g}, first bad {np.argwhere(bad)[:3].tolist()}")


def tight_errors(got, ref_f):
    """Errors in fp16 ulps of the outputs the tight bar covers (see the module docstring)."""
    got = np.asarray(got, dtype=np.float64)
    ref_f = np.asarray(ref_f, dtype=np.float64)
    big = np.abs(ref_f) >= TIGHT_FLOOR * np.abs(ref_f).max()
    return np.abs(got - ref_f)[big] / fp16_ulp(ref_f[big])


def assert_tight(got, ref_f, what=""):
    e = tight_errors(got, ref_f)
    if e.size == 0:
        return
    assert e.max() <= TIGHT_ULP, (f"{what}: {int((e > TIGHT_ULP).sum())}/{e.size} outputs beyond {TIGHT_ULP} ulp of "
                                  f"the binary32-unfold oracle rounded to fp16, max {e.max():.3f} ulp")
    assert e.mean() <= TIGHT_MEAN_ULP, f"{what}: mean error {e.mean():.3f} ulp over {e.size} outputs"


def assert_matches(got, ref_d, ref_f, what=""):
    """Both bars: the stated one against the binary64 and the binary32-unfold oracle, the tight one against the
    binary32-unfold oracle."""
    assert_within_tolerance(got, ref_d, f"{what} (binary64 oracle)")
    assert_within_tolerance(got, ref_f, f"{what} (binary32-unfold oracle)")
    assert_tight(got, ref_f, what)
