"""The exactness arguments the CUDA kernels rest on, checked exhaustively on the host (no GPU, no library).

Each is a fact of integer or binary32 arithmetic that a kernel uses in place of the plain step it stands for
(method: WeightQuantBatchMatmulExperiment page, section 4.1, steps 9-10); the GPU parity tests check the kernels
themselves, these check that the substitutions cannot lose anything on any input:
  - decode products: per 32-bit weight word, dp4a of the low nibbles against 16 A_lo - A_hi plus dp4a of the whole
    word against A_hi is 16 times the word's exact contribution to Y_i, and 16 A_lo - A_hi fits int8;
  - the int -> float conversion by a 1.5 * 2^23 bias is exact for |v| < 2^22, which covers every dot product;
  - offset-binary nibble bytes u = w + 8 read as E4M3 are u * 2^-9 exactly (bytes 0-7 subnormal, 8-15 normal).
"""
import numpy as np

PLANE = np.arange(-7, 8)          # |A_i| <= 7: A_i = rint of a value in [-7.49, 7.49]
NIBBLE = np.arange(16)            # u = w + 8 for int4 w in [-8, 7]


def test_decode_recoding_is_exact_for_every_byte_lane():
    # one byte lane of a weight word: low nibble lo (k), high nibble hi (k + 4), plane values a_lo, a_hi
    lo, hi, a_lo, a_hi = np.meshgrid(NIBBLE, NIBBLE, PLANE, PLANE, indexing="ij")
    d = 16 * a_lo - a_hi
    assert d.min() >= -128 and d.max() <= 127                    # stored as int8
    byte = lo + 16 * hi                                           # the whole word's byte, unsigned
    assert byte.min() >= 0 and byte.max() <= 255
    got = lo * d + byte * a_hi                                    # the two dp4a terms of this byte lane
    assert np.array_equal(got, 16 * (lo * a_lo + hi * a_hi))


def test_decode_recoding_sums_over_a_word_and_a_chunk():
    # the identity is per byte lane, so any sum of lanes keeps it: a 32-k chunk (four words), random values
    rng = np.random.default_rng(11)
    for _ in range(200):
        u = rng.integers(0, 16, size=32)                          # k = 8q + b (low) and 8q + 4 + b (high)
        a = rng.integers(-7, 8, size=32)
        words = u.reshape(4, 2, 4)                                # [word q][half][byte b]
        planes = a.reshape(4, 2, 4)
        lo, hi = words[:, 0], words[:, 1]
        d, h = 16 * planes[:, 0] - planes[:, 1], planes[:, 1]
        dot = int((lo * d).sum() + ((lo + 16 * hi) * h).sum())
        assert dot == 16 * int((a * u).sum())


def test_dot_products_stay_inside_the_exact_conversion_range():
    # the largest |16 sum A u| over one 32-k chunk, and over a whole 128-k group as the debug path adds them
    assert 16 * 7 * 15 * 32 < 2 ** 22
    assert 16 * 7 * 15 * 128 < 2 ** 22


def test_bias_conversion_is_exact_below_2_pow_22():
    v = np.arange(-(2 ** 22) + 1, 2 ** 22, dtype=np.int64)
    bits = (v + 0x4B400000).astype(np.uint32)
    as_float = bits.view(np.float32)
    got = as_float - np.float32(12582912.0)                       # 1.5 * 2^23, one binary32 subtraction
    assert got.dtype == np.float32
    assert np.array_equal(got.astype(np.int64), v)


def e4m3_value(byte):
    """OCP FP8 E4M3 (bias 7, no infinities): sign, 4 exponent bits, 3 mantissa bits."""
    sign = -1.0 if byte & 0x80 else 1.0
    e, m = (byte >> 3) & 0xF, byte & 0x7
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** (1 - 7)
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def test_nibble_bytes_are_exact_e4m3_multiples_of_2_pow_minus_9():
    for u in NIBBLE:
        assert e4m3_value(int(u)) == float(u) * 2.0 ** -9
    # and the largest MMA-unit product the path forms stays exact in binary32: 2^-9 * 15 * 7 * K-group of 128
    assert (15 * 7 * 128) < 2 ** 24
