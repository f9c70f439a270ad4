"""The oracle's pins must bite: plant a plausible mistake in a copy of the oracle's C source and check that at
least one pin of test_oracle_pins.py rejects the mutated copy. Mistakes are planted on the CPU, in the oracle only.
"""
import os

import pytest

import oracle
import test_oracle_pins as P
import test_oracle_w8 as W
import test_oracle_zp_bias as Z

SRC = os.path.join(os.path.dirname(oracle.__file__), "wqbmm_oracle.c")

# (name, text in the source, replacement)
MUTATIONS = [
    ("second factor 7.49 instead of 14.98 (binary64)", "double tmp2 = (tmp1 - A1) * 14.98;",
     "double tmp2 = (tmp1 - A1) * 7.49;"),
    ("second factor 7.49f instead of 14.98f (binary32)", "float tmp2 = d1 * f2;", "float tmp2 = d1 * f1;"),
    ("residual sign flipped", "double tmp2 = (tmp1 - A1) * 14.98;", "double tmp2 = (A1 - tmp1) * 14.98;"),
    ("third residual from the wrong plane", "double tmp3 = (tmp2 - A2) * 14.98;",
     "double tmp3 = (tmp2 - A1) * 14.98;"),
    ("round half away from zero (binary32)", "float A3 = rintf(tmp3);", "float A3 = roundf(tmp3);"),
    ("A_max without the absolute value", "double v = fabs(oracle_half_to_double(xg[k]));",
     "double v = oracle_half_to_double(xg[k]);"),
    ("third plane dropped from the combine", " + y3 / (7.49 * 14.98 * 14.98))", ")"),
    ("middle divisor 14.98 instead of 7.49*14.98", "y2 / (7.49 * 14.98)", "y2 / (14.98)"),
    ("A_max left out of the combine", "* amax\n", "\n"),
    ("scale of the neighbouring group", "sc[n] = oracle_half_to_double(scale[g * N + n]);",
     "sc[n] = oracle_half_to_double(scale[((g + 1) % Gn) * N + n]);"),
    ("groups overwrite instead of accumulate", "yr[n] = ygroup + yr[n];", "yr[n] = ygroup;"),
    ("nibble order swapped", "w[(2 * kk) * N + n] = (int8_t)(lo >= 8 ? lo - 16 : lo);",
     "w[(2 * kk) * N + n] = (int8_t)(hi >= 8 ? hi - 16 : hi);"),
    ("int4 read as unsigned", "(int8_t)(hi >= 8 ? hi - 16 : hi)", "(int8_t)(hi)"),
    ("weight rows of a group reversed", "const int8_t *row = wg + k * N;", "const int8_t *row = wg + (G - 1 - k) * N;"),
    ("fp16 exponent bias off by one", "v = ldexp(1024.0 + f, e - 25);", "v = ldexp(1024.0 + f, e - 24);"),
    ("zero point added instead of subtracted", "double y1 = yi[n] - z * s1", "double y1 = yi[n] + z * s1"),
    ("zero point times the wrong plane sum", "s2 += a[G + k];", "s2 += a[k];"),
    ("bias dropped", "yr[n] = yr[n] + oracle_half_to_double(bias[n]);", "yr[n] = yr[n];"),
    ("int8 weights of the wrong group", "w8 + g * G * N, G, N, yi", "w8 + g * N, G, N, yi"),
    ("int8 weight read as unsigned", "const int8_t *row = w8 + k * N;",
     "const uint8_t *row = (const uint8_t *)w8 + k * N;"),
]

PINS = [
    lambda o: P.test_half_decode_all_bit_patterns(o),
    lambda o: P.test_int4_decode_hand_fixture(o),
    lambda o: P.test_worked_unfold_values(o),
    lambda o: P.test_binary32_ties_round_half_even(o),
    lambda o: P.test_plane_bound_and_reconstruction(o, "normal", 1.0, 64),
    lambda o: P.test_hand_2x2(o),
    lambda o: P.test_hand_4x4_two_groups(o),
    lambda o: P.test_msd_within_closed_form_bound_of_direct_matmul(o, "normal", "u8", 128),
    lambda o: P.test_identity_weights_return_x(o),
    lambda o: P.test_constant_groups_scale_column_sums(o),
    lambda o: P.test_group_and_column_permutation_invariance(o),
    lambda o: Z.test_integer_zero_point_equals_shifted_weights(o, oracle.MODE_D, 1),
    lambda o: Z.test_bias_adds_itself(o),
    lambda o: W.test_w8_in_int4_range_is_the_int4_path(o, oracle.MODE_D),
    lambda o: W.test_w8_within_closed_form_bound(o, oracle.MODE_D),
]


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(source, tmp_path, name, old, new):
    assert source.count(old) >= 1, f"mutation anchor not found: {old!r}"
    lib = oracle.build_variant(source.replace(old, new, 1), str(tmp_path), "mutant")
    mutant = oracle.Oracle(lib)
    caught = []
    for pin in PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError):
            caught.append(pin)
    assert caught, f"no pin rejects the planted mistake: {name}"


def test_unmutated_copy_passes_every_pin(source, tmp_path):
    lib = oracle.build_variant(source, str(tmp_path), "copy")
    copy = oracle.Oracle(lib)
    for pin in PINS:
        pin(copy)
