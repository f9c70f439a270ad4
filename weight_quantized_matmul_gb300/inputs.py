"""Seeded synthetic inputs for the A16W4 per-group MSD matmul.

This module only draws random numbers and lays them out in the operator's input formats. It holds none of the
method's arithmetic (no A_max, no residual unfold, no matmul, no scale combine), so the CUDA path and the CPU
oracle can both be fed from it without sharing any of the computation under test.

Input formats (WeightQuantBatchMatmulExperiment page, section 4.2 operator spec and section 4.3 sample data):
  x      fp16 [M, K], row-major
  w      signed int4 [K, N], packed two per byte along K into uint8 [K/2, N]: byte (kk, n) holds w[2kk, n] in its
         low nibble and w[2kk+1, n] in its high nibble, two's complement
  scale  fp16 [K/G, N] (antiquant_scale, one row per K-group)

Random numbers come from SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
OOPSLA 2014) evaluated at counter positions: value(i) = mix(key + (i + 1) * GAMMA). Every element can be
regenerated on its own, and the streams are identical on every platform and numpy version.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import Optional

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function on a uint64 array (wrapping arithmetic)."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        base = np.array([(int(seed) << 20) ^ int(stream)], dtype=np.uint64)
        return _mix(base * _GAMMA + _GAMMA)[0]


def raw_u64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """`count` SplitMix64 outputs of (seed, stream) at counters start .. start+count-1."""
    key = _key(seed, stream)
    idx = np.arange(start, start + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + (idx + np.uint64(1)) * _GAMMA)


def _u24(z: np.ndarray) -> np.ndarray:
    """Top 24 bits as a float64 in [0, 1)."""
    return (z >> np.uint64(40)).astype(np.float64) * (1.0 / (1 << 24))


def uniform(seed: int, stream: int, count: int, lo: float, hi: float) -> np.ndarray:
    out = np.empty(count, dtype=np.float64)
    for s in range(0, count, _CHUNK):
        c = min(_CHUNK, count - s)
        out[s:s + c] = lo + (hi - lo) * _u24(raw_u64(seed, stream, s, c))
    return out


def normal(seed: int, stream: int, count: int) -> np.ndarray:
    """Standard normals by Box-Muller; element i uses counters 2i and 2i+1."""
    out = np.empty(count, dtype=np.float64)
    for s in range(0, count, _CHUNK):
        c = min(_CHUNK, count - s)
        z = raw_u64(seed, stream, 2 * s, 2 * c)
        u1 = ((z[0::2] >> np.uint64(40)).astype(np.float64) + 1.0) * (1.0 / (1 << 24))  # (0, 1]
        u2 = _u24(z[1::2])
        out[s:s + c] = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return out


def student_t3(seed: int, stream: int, count: int) -> np.ndarray:
    """Student-t with 3 degrees of freedom: Z0 / sqrt((Z1^2 + Z2^2 + Z3^2) / 3), four independent normals."""
    z = normal(seed, stream, 4 * count).reshape(count, 4)
    chi2 = (z[:, 1:] ** 2).sum(axis=1)
    return z[:, 0] / np.sqrt(chi2 / 3.0)


def int_uniform(seed: int, stream: int, count: int, lo: int, hi: int) -> np.ndarray:
    """Integers uniform on [lo, hi] by Lemire's multiply-shift on 32 random bits (bias below 2^-28)."""
    span = np.uint64(hi - lo + 1)
    out = np.empty(count, dtype=np.int16)
    for s in range(0, count, _CHUNK):
        c = min(_CHUNK, count - s)
        z = raw_u64(seed, stream, s, c) >> np.uint64(32)
        out[s:s + c] = ((z * span) >> np.uint64(32)).astype(np.int64) + lo
    return out


def pack_int4_along_k(w: np.ndarray) -> np.ndarray:
    """int [K, N] in [-8, 7] -> uint8 [K/2, N]; low nibble = even k, high nibble = odd k (two's complement)."""
    K, N = w.shape
    if K % 2:
        raise ValueError("K must be even to pack two int4 per byte along K")
    lo = (w[0::2].astype(np.int16) & 0xF).astype(np.uint8)
    hi = (w[1::2].astype(np.int16) & 0xF).astype(np.uint8)
    return lo | (hi << 4)


def fp16(a: np.ndarray) -> np.ndarray:
    """Round to IEEE binary16, nearest-even (numpy's float64 -> float16 conversion)."""
    return np.asarray(a, dtype=np.float64).astype(np.float16)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    K: int
    N: int
    G: int
    seed: int
    x_dist: str            # "normal", "normal_cols20", "t3_clip60", "uniform3"
    x_sigma: float
    w_dist: str            # "u8" (uniform [-8,7]), "pm1_mix" (p=.5 in {-1,1} else uniform [-8,7]), "u7" ([-7,7])
    scale_lo: float
    scale_hi: float
    sample_rows: int = 0   # >0: the oracle checks this many seeded rows (always rows 0 and M-1)

    @property
    def groups(self) -> int:
        return self.K // self.G

    def algorithmic_bytes(self) -> int:
        """HBM bytes one call must move: x 2MK + packed W KN/2 + scale 2(K/G)N + y 2MN."""
        return 2 * self.M * self.K + self.K * self.N // 2 + 2 * self.groups * self.N + 2 * self.M * self.N

    def weight_bytes(self) -> int:
        return self.K * self.N // 2

    def int8_equiv_ops(self) -> int:
        """3 planes x 2 ops per multiply-add x M N K."""
        return 6 * self.M * self.N * self.K


# The five measurement shapes (decode, small-batch, mid-batch and prefill regimes) plus the operator page's own
# sample shape (section 4.3: M=1, N=12288, K=8192, groupSize=128, x and scale U[-3,3], weights in [-7,7]).
WORKLOADS = {
    "pr1_m16_k1024_n1024": Workload("pr1_m16_k1024_n1024", 16, 1024, 1024, 128, 0, "normal", 1.0, "u8", 0.005, 0.02),
    "decode_m1_k4096_n4096": Workload("decode_m1_k4096_n4096", 1, 4096, 4096, 128, 1, "normal", 1.0, "u8",
                                      0.005, 0.02),
    "ffn_up_m8_k4096_n11008": Workload("ffn_up_m8_k4096_n11008", 8, 4096, 11008, 128, 2, "t3_clip60", 1.0, "u8",
                                       0.002, 0.03),
    "mid_m128_k5120_n13824": Workload("mid_m128_k5120_n13824", 128, 5120, 13824, 128, 3, "normal_cols20", 1.0,
                                      "pm1_mix", 0.005, 0.02),
    "prefill_m2048_k8192_n28672": Workload("prefill_m2048_k8192_n28672", 2048, 8192, 28672, 64, 4, "normal", 0.5,
                                           "u8", 0.001, 0.01, sample_rows=64),
    "page_sample_m1_k8192_n12288": Workload("page_sample_m1_k8192_n12288", 1, 8192, 12288, 128, 5, "uniform3", 3.0,
                                            "u7", -3.0, 3.0),
}

# stream ids
_S_X, _S_W, _S_SCALE, _S_COLS, _S_WSEL, _S_WPM, _S_ROWS, _S_ZP, _S_BIAS, _S_W8 = 1, 2, 3, 4, 5, 6, 7, 8, 9, 10


def make_x(wl: Workload, M: Optional[int] = None) -> np.ndarray:
    M = wl.M if M is None else M
    n = M * wl.K
    if wl.x_dist == "normal":
        v = wl.x_sigma * normal(wl.seed, _S_X, n)
    elif wl.x_dist == "normal_cols20":
        v = normal(wl.seed, _S_X, n).reshape(M, wl.K)
        v[:, outlier_columns(wl)] *= 20.0
        v = v.reshape(-1)
    elif wl.x_dist == "t3_clip60":
        v = np.clip(student_t3(wl.seed, _S_X, n), -60.0, 60.0)
    elif wl.x_dist == "uniform3":
        v = uniform(wl.seed, _S_X, n, -3.0, 3.0)
    else:
        raise ValueError(wl.x_dist)
    return fp16(v).reshape(M, wl.K)


def outlier_columns(wl: Workload) -> np.ndarray:
    """floor(1% of K) columns picked by a seeded shuffle (the 'scaled x20' activation outliers)."""
    count = (wl.K * 1) // 100
    keys = raw_u64(wl.seed, _S_COLS, 0, wl.K)
    return np.sort(np.argsort(keys, kind="stable")[:count])


def make_w_packed(wl: Workload) -> np.ndarray:
    K, N = wl.K, wl.N
    if wl.w_dist == "u8":
        # 4 random bits per nibble are uniform on [-8, 7] read as two's complement; 8 bytes per SplitMix64 draw
        nbytes = (K // 2) * N
        out = np.empty(nbytes, dtype=np.uint8)
        step = _CHUNK * 8
        for s in range(0, nbytes, step):
            c = min(step, nbytes - s)
            z = raw_u64(wl.seed, _S_W, s // 8, (c + 7) // 8)
            out[s:s + c] = z.astype("<u8").view(np.uint8)[:c]
        return out.reshape(K // 2, N)
    w = make_w_int(wl)
    return pack_int4_along_k(w)


def make_w_int(wl: Workload) -> np.ndarray:
    """Element-wise int4 weights [K, N] as int8, for the distributions that are not plain uniform nibbles."""
    K, N = wl.K, wl.N
    n = K * N
    if wl.w_dist == "u7":
        return int_uniform(wl.seed, _S_W, n, -7, 7).astype(np.int8).reshape(K, N)
    if wl.w_dist == "pm1_mix":
        out = np.empty(n, dtype=np.int8)
        for s in range(0, n, _CHUNK):
            c = min(_CHUNK, n - s)
            sel = raw_u64(wl.seed, _S_WSEL, s, c) >> np.uint64(63)           # 1 bit: which branch
            sign = raw_u64(wl.seed, _S_WPM, s, c) >> np.uint64(63)           # 1 bit: -1 or +1
            uni = (raw_u64(wl.seed, _S_W, s, c) >> np.uint64(60)).astype(np.int16)  # 4 bits: [-8, 7]
            uni = np.where(uni >= 8, uni - 16, uni)
            pm1 = np.where(sign == 1, 1, -1)
            out[s:s + c] = np.where(sel == 1, pm1, uni).astype(np.int8)
        return out.reshape(K, N)
    raise ValueError(wl.w_dist)


def make_scale(wl: Workload) -> np.ndarray:
    n = wl.groups * wl.N
    return fp16(uniform(wl.seed, _S_SCALE, n, wl.scale_lo, wl.scale_hi)).reshape(wl.groups, wl.N)


def make_zero_point(wl: Workload, kind: str = "int") -> np.ndarray:
    """Zero points fp16 [K/G, N] of asymmetric weights (the weight stands for (w - zp) * scale): "int" draws
    integers in [-4, 4], "frac" uniform reals in [-4, 4] rounded to fp16."""
    n = wl.groups * wl.N
    if kind == "int":
        z = int_uniform(wl.seed, _S_ZP, n, -4, 4).astype(np.float64)
    elif kind == "frac":
        z = uniform(wl.seed, _S_ZP, n, -4.0, 4.0)
    else:
        raise ValueError(kind)
    return fp16(z).reshape(wl.groups, wl.N)


def make_w8(wl: Workload) -> np.ndarray:
    """Int8 weights [K, N] uniform on [-128, 127] (W8)."""
    return int_uniform(wl.seed, _S_W8, wl.K * wl.N, -128, 127).astype(np.int8).reshape(wl.K, wl.N)


def make_bias(wl: Workload, lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    """Bias fp16 [N], uniform in [lo, hi]."""
    return fp16(uniform(wl.seed, _S_BIAS, wl.N, lo, hi))


def make_inputs(wl: Workload):
    """(x fp16 [M,K], w_packed uint8 [K/2,N], scale fp16 [K/G,N])."""
    return make_x(wl), make_w_packed(wl), make_scale(wl)


def sample_rows(wl: Workload, count: Optional[int] = None) -> np.ndarray:
    """Seeded row sample for oracle checks at full size: rows 0 and M-1 always, the rest by a seeded shuffle."""
    count = wl.sample_rows if count is None else count
    if count <= 0 or count >= wl.M:
        return np.arange(wl.M, dtype=np.int64)
    keys = raw_u64(wl.seed, _S_ROWS, 0, wl.M)
    order = [int(r) for r in np.argsort(keys, kind="stable") if r not in (0, wl.M - 1)]
    rows = sorted({0, wl.M - 1, *order[:count - 2]})
    return np.asarray(rows, dtype=np.int64)


def digest(*arrays: np.ndarray) -> str:
    """Short content hash of input buffers, for logging which inputs a run used."""
    h = hashlib.sha256()
    for a in arrays:
        h.update(np.ascontiguousarray(a).view(np.uint8).tobytes())
    return h.hexdigest()[:16]


def small_case(M: int, K: int, N: int, G: int, seed: int, x_dist: str = "normal", w_dist: str = "u8",
               scale_lo: float = 0.005, scale_hi: float = 0.02, x_sigma: float = 1.0) -> Workload:
    """An ad-hoc shape with one of the workload distributions (parity tests at sizes the oracle finishes fast)."""
    return Workload(f"case_m{M}_k{K}_n{N}_g{G}_s{seed}", M, K, N, G, seed, x_dist, x_sigma, w_dist,
                    scale_lo, scale_hi)
