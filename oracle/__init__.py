"""ctypes front end of the CPU oracle (test infrastructure only).

Only the tests, `__graft_entry__.smoke()` and the benchmark's CPU-baseline leg may import this package. The
library's product path never calls it. The C source (`wqbmm_oracle.c`) states the method and the readings it takes;
this file only marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

MODE_D = 0   # unfold in binary64 with the decimal constants 7.49 and 14.98
MODE_F = 1   # unfold in binary32 with 7.49f and 14.98f, each operation rounded

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wqbmm_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math", "-fexcess-precision=standard"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction, IEEE semantics). Returns the library path."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _bind(path: str):
    lib = ctypes.CDLL(path)
    i64, p = ctypes.c_int64, ctypes.c_void_p
    lib.oracle_half_to_double.restype = ctypes.c_double
    lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_decode_int4.argtypes = [p, i64, i64, p]
    lib.oracle_unfold.argtypes = [p, i64, i64, i64, ctypes.c_int, p, p]
    lib.oracle_group_partials.argtypes = [p, p, i64, i64, i64, i64, i64, ctypes.c_int, p, i64, p]
    lib.oracle_msd_rows.argtypes = [p, p, p, i64, i64, i64, i64, ctypes.c_int, p, i64, p]
    lib.oracle_direct_rows.argtypes = [p, p, p, i64, i64, i64, i64, p, i64, p]
    lib.oracle_msd_rows_ex.argtypes = [p, p, p, p, p, i64, i64, i64, i64, ctypes.c_int, p, i64, p]
    lib.oracle_direct_rows_ex.argtypes = [p, p, p, p, p, i64, i64, i64, i64, p, i64, p]
    lib.oracle_msd_rows_w8.argtypes = [p, p, p, p, p, i64, i64, i64, i64, ctypes.c_int, p, i64, p]
    lib.oracle_direct_rows_w8.argtypes = [p, p, p, p, p, i64, i64, i64, i64, p, i64, p]
    for f in ("oracle_decode_int4", "oracle_unfold", "oracle_group_partials", "oracle_msd_rows",
              "oracle_direct_rows", "oracle_msd_rows_ex", "oracle_direct_rows_ex", "oracle_msd_rows_w8",
              "oracle_direct_rows_w8"):
        getattr(lib, f).restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"{what}: oracle error {rc}")


def _as_half_bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        return x.view(np.uint16)
    if x.dtype == np.uint16:
        return x
    raise TypeError("expected float16 data")


def _rows(M: int, rows) -> np.ndarray:
    if rows is None:
        return np.arange(M, dtype=np.int64)
    return np.ascontiguousarray(np.asarray(rows, dtype=np.int64))


class Oracle:
    """The oracle's functions bound to one compiled copy of the C source (the default build, or another one)."""

    def __init__(self, path: str = ""):
        self._path = path
        self._own = None

    def _lib(self):
        if not self._path:
            return _load()
        if self._own is None:
            self._own = _bind(self._path)
        return self._own

    def half_to_double(self, bits: int) -> float:
        return self._lib().oracle_half_to_double(int(bits))

    def decode_int4(self, w_packed: np.ndarray, K: int, N: int) -> np.ndarray:
        w_packed = np.ascontiguousarray(w_packed, dtype=np.uint8)
        out = np.empty((K, N), dtype=np.int8)
        _check(self._lib().oracle_decode_int4(_ptr(w_packed), K, N, _ptr(out)), "decode_int4")
        return out

    def unfold(self, x: np.ndarray, G: int, mode: int = MODE_F):
        """Steps 1-8: (planes int8 [3, M, K], amax float64 [M, K/G])."""
        xb = _as_half_bits(x)
        M, K = xb.shape
        planes = np.empty((3, M, K), dtype=np.int8)
        amax = np.empty((M, K // G), dtype=np.float64)
        _check(self._lib().oracle_unfold(_ptr(xb), M, K, G, mode, _ptr(planes), _ptr(amax)), "unfold")
        return planes, amax

    def group_partials(self, x: np.ndarray, w_packed: np.ndarray, N: int, G: int, g: int, mode: int = MODE_F,
                       rows=None):
        """Step 9 for group g: int32 [3, len(rows), N]."""
        xb = _as_half_bits(x)
        M, K = xb.shape
        w_packed = np.ascontiguousarray(w_packed, dtype=np.uint8)
        r = _rows(M, rows)
        out = np.empty((3, len(r), N), dtype=np.int32)
        _check(self._lib().oracle_group_partials(_ptr(xb), _ptr(w_packed), M, K, N, G, g, mode, _ptr(r), len(r),
                                                 _ptr(out)), "group_partials")
        return out

    def msd_matmul(self, x: np.ndarray, w_packed: np.ndarray, scale: np.ndarray, G: int, mode: int = MODE_D,
                   rows=None):
        """Steps 1-11: float64 [len(rows), N]."""
        xb = _as_half_bits(x)
        sb = _as_half_bits(scale)
        M, K = xb.shape
        N = sb.shape[1]
        w_packed = np.ascontiguousarray(w_packed, dtype=np.uint8)
        r = _rows(M, rows)
        out = np.empty((len(r), N), dtype=np.float64)
        _check(self._lib().oracle_msd_rows(_ptr(xb), _ptr(w_packed), _ptr(sb), M, K, N, G, mode, _ptr(r), len(r),
                                           _ptr(out)), "msd_matmul")
        return out

    def msd_matmul_ex(self, x: np.ndarray, w_packed: np.ndarray, scale: np.ndarray, G: int, zero_point=None,
                      bias=None, mode: int = MODE_D, rows=None):
        """Steps 1-11 with optional zero points fp16 [K/G, N] (weights stand for (w - zp) * scale) and bias fp16 [N]:
        float64 [len(rows), N]."""
        xb = _as_half_bits(x)
        sb = _as_half_bits(scale)
        zb = None if zero_point is None else _as_half_bits(zero_point)
        bb = None if bias is None else _as_half_bits(np.asarray(bias).reshape(-1))
        M, K = xb.shape
        N = sb.shape[1]
        w_packed = np.ascontiguousarray(w_packed, dtype=np.uint8)
        r = _rows(M, rows)
        out = np.empty((len(r), N), dtype=np.float64)
        _check(self._lib().oracle_msd_rows_ex(_ptr(xb), _ptr(w_packed), _ptr(sb),
                                              None if zb is None else _ptr(zb), None if bb is None else _ptr(bb),
                                              M, K, N, G, mode, _ptr(r), len(r), _ptr(out)), "msd_matmul_ex")
        return out

    def direct_matmul_ex(self, x: np.ndarray, w_packed: np.ndarray, scale: np.ndarray, G: int, zero_point=None,
                         bias=None, rows=None):
        """x . ((w - zp) * scale) + bias in binary64: float64 [len(rows), N]."""
        xb = _as_half_bits(x)
        sb = _as_half_bits(scale)
        zb = None if zero_point is None else _as_half_bits(zero_point)
        bb = None if bias is None else _as_half_bits(np.asarray(bias).reshape(-1))
        M, K = xb.shape
        N = sb.shape[1]
        w_packed = np.ascontiguousarray(w_packed, dtype=np.uint8)
        r = _rows(M, rows)
        out = np.empty((len(r), N), dtype=np.float64)
        _check(self._lib().oracle_direct_rows_ex(_ptr(xb), _ptr(w_packed), _ptr(sb),
                                                 None if zb is None else _ptr(zb), None if bb is None else _ptr(bb),
                                                 M, K, N, G, _ptr(r), len(r), _ptr(out)), "direct_matmul_ex")
        return out

    def msd_matmul_w8(self, x: np.ndarray, w8: np.ndarray, scale: np.ndarray, G: int, zero_point=None, bias=None,
                      mode: int = MODE_D, rows=None):
        """Steps 1-11 with int8 weights w8 [K, N] (and optional zero points / bias): float64 [len(rows), N]."""
        xb = _as_half_bits(x)
        sb = _as_half_bits(scale)
        zb = None if zero_point is None else _as_half_bits(zero_point)
        bb = None if bias is None else _as_half_bits(np.asarray(bias).reshape(-1))
        M, K = xb.shape
        N = sb.shape[1]
        w8 = np.ascontiguousarray(w8, dtype=np.int8)
        assert w8.shape == (K, N)
        r = _rows(M, rows)
        out = np.empty((len(r), N), dtype=np.float64)
        _check(self._lib().oracle_msd_rows_w8(_ptr(xb), _ptr(w8), _ptr(sb), None if zb is None else _ptr(zb),
                                              None if bb is None else _ptr(bb), M, K, N, G, mode, _ptr(r), len(r),
                                              _ptr(out)), "msd_matmul_w8")
        return out

    def direct_matmul_w8(self, x: np.ndarray, w8: np.ndarray, scale: np.ndarray, G: int, zero_point=None,
                         bias=None, rows=None):
        """x . ((w8 - zp) * scale) + bias in binary64: float64 [len(rows), N]."""
        xb = _as_half_bits(x)
        sb = _as_half_bits(scale)
        zb = None if zero_point is None else _as_half_bits(zero_point)
        bb = None if bias is None else _as_half_bits(np.asarray(bias).reshape(-1))
        M, K = xb.shape
        N = sb.shape[1]
        w8 = np.ascontiguousarray(w8, dtype=np.int8)
        assert w8.shape == (K, N)
        r = _rows(M, rows)
        out = np.empty((len(r), N), dtype=np.float64)
        _check(self._lib().oracle_direct_rows_w8(_ptr(xb), _ptr(w8), _ptr(sb), None if zb is None else _ptr(zb),
                                                 None if bb is None else _ptr(bb), M, K, N, G, _ptr(r), len(r),
                                                 _ptr(out)), "direct_matmul_w8")
        return out

    def direct_matmul(self, x: np.ndarray, w_packed: np.ndarray, scale: np.ndarray, G: int, rows=None):
        """x . (w * scale) in binary64: float64 [len(rows), N]."""
        xb = _as_half_bits(x)
        sb = _as_half_bits(scale)
        M, K = xb.shape
        N = sb.shape[1]
        w_packed = np.ascontiguousarray(w_packed, dtype=np.uint8)
        r = _rows(M, rows)
        out = np.empty((len(r), N), dtype=np.float64)
        _check(self._lib().oracle_direct_rows(_ptr(xb), _ptr(w_packed), _ptr(sb), M, K, N, G, _ptr(r), len(r),
                                              _ptr(out)), "direct_matmul")
        return out


def build_variant(source_text: str, out_dir: str, name: str) -> str:
    """Compile C source text with the oracle's flags into out_dir/name.so (used to check that the pins bite)."""
    src = os.path.join(out_dir, name + ".c")
    lib = os.path.join(out_dir, name + ".so")
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", *_CFLAGS, "-o", lib, src, "-lm"], check=True)
    return lib


_default = Oracle()
half_to_double = _default.half_to_double
decode_int4 = _default.decode_int4
unfold = _default.unfold
group_partials = _default.group_partials
msd_matmul = _default.msd_matmul
direct_matmul = _default.direct_matmul
msd_matmul_ex = _default.msd_matmul_ex
direct_matmul_ex = _default.direct_matmul_ex
msd_matmul_w8 = _default.msd_matmul_w8
direct_matmul_w8 = _default.direct_matmul_w8
