"""A16W4 per-group pseudo-quantized matmul by MSD for GB300 (sm_103a).

Python binding of the C ABI declared in include/wqbmm.h. Every function here only marshals arguments (torch tensors
or raw device pointers, sizes, a stream) and calls the library of the same name; all arithmetic runs in the CUDA
kernels of libwqbmm.so. There is no fallback: if the library is missing or the device is not a GB300, calls raise.
PyTorch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "WqbmmError", "library_path", "load_library", "wqbmm_prepacked_weight_bytes", "wqbmm_prepack_weight",
    "wqbmm_workspace_bytes", "wqbmm_run", "wqbmm_debug_unfold", "wqbmm_debug_group_partials",
    "wqbmm_read_device_status", "wqbmm_debug_wait_timeout", "wqbmm_status_string", "prepack_weight",
    "allocate_workspace", "msd_matmul", "SYMBOLS", "wqbmm_run_static_scratch", "wqbmm_prepack_weight_nk",
    "prepack_weight_nk", "wqbmm_run_ex", "wqbmm_run_batched", "wqbmm_prepacked_weight_bytes_w8",
    "wqbmm_prepack_weight_w8", "wqbmm_workspace_bytes_w8", "wqbmm_run_w8", "prepack_weight_w8", "msd_matmul_w8",
    "wqbmm_run_part",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libwqbmm.so")
_lock = threading.Lock()
_lib = None

OK, ERR_NULLPTR, ERR_INVALID, ERR_UNSUPPORTED_ARCH, ERR_CUDA, ERR_DEVICE_TIMEOUT, ERR_SCRATCH_LIMIT = range(7)

# every entry point include/wqbmm.h declares
SYMBOLS = (
    "wqbmm_prepacked_weight_bytes", "wqbmm_prepack_weight", "wqbmm_workspace_bytes", "wqbmm_run",
    "wqbmm_debug_unfold", "wqbmm_debug_group_partials", "wqbmm_read_device_status", "wqbmm_debug_wait_timeout",
    "wqbmm_status_string", "wqbmm_run_static_scratch", "wqbmm_prepack_weight_nk", "wqbmm_run_ex",
    "wqbmm_run_batched", "wqbmm_prepacked_weight_bytes_w8", "wqbmm_prepack_weight_w8", "wqbmm_workspace_bytes_w8",
    "wqbmm_run_w8", "wqbmm_run_part",
)


class WqbmmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {wqbmm_status_string(status)} (status {status})")


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """The loaded libwqbmm.so (built in-tree by __graft_entry__.build())."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(f"{_LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; "
                                   f"g.build()\"`")
            lib = ctypes.CDLL(_LIB_PATH)
            i64, p, sz = ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
            st = ctypes.c_int
            sig = {
                "wqbmm_prepacked_weight_bytes": [i64, i64, i64, ctypes.POINTER(sz)],
                "wqbmm_prepack_weight": [p, p, i64, i64, i64, p],
                "wqbmm_workspace_bytes": [i64, i64, i64, i64, ctypes.POINTER(sz)],
                "wqbmm_run": [p, p, p, p, i64, i64, i64, i64, p, sz, p],
                "wqbmm_run_ex": [p, p, p, p, p, p, i64, i64, i64, i64, p, sz, p],
                "wqbmm_run_part": [p, p, p, p, p, p, i64, i64, i64, i64, p, sz, ctypes.c_int, p],
                "wqbmm_run_batched": [p, p, p, p, p, p, i64, i64, i64, i64, i64, i64, i64, p, sz, p],
                "wqbmm_prepacked_weight_bytes_w8": [i64, i64, i64, ctypes.POINTER(sz)],
                "wqbmm_prepack_weight_w8": [p, p, i64, i64, i64, p],
                "wqbmm_workspace_bytes_w8": [i64, i64, i64, i64, ctypes.POINTER(sz)],
                "wqbmm_run_w8": [p, p, p, p, p, p, i64, i64, i64, i64, p, sz, p],
                "wqbmm_debug_unfold": [p, i64, i64, i64, p, p, p],
                "wqbmm_debug_group_partials": [p, p, i64, i64, i64, i64, i64, p, p, sz, p],
                "wqbmm_read_device_status": [ctypes.POINTER(ctypes.c_int32), ctypes.c_int, p],
                "wqbmm_debug_wait_timeout": [i64, p],
                "wqbmm_run_static_scratch": [p, p, p, p, i64, i64, i64, i64, p],
                "wqbmm_prepack_weight_nk": [p, p, i64, i64, i64, p],
            }
            for name, args in sig.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = st
            lib.wqbmm_status_string.argtypes = [st]
            lib.wqbmm_status_string.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def _ptr(a) -> int | None:
    if a is None:
        return None
    if isinstance(a, int):
        return a
    return a.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, where: str):
    if status != OK:
        raise WqbmmError(status, where)


def wqbmm_status_string(status: int) -> str:
    return load_library().wqbmm_status_string(int(status)).decode()


def wqbmm_prepacked_weight_bytes(K: int, N: int, G: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load_library().wqbmm_prepacked_weight_bytes(K, N, G, ctypes.byref(out)), "wqbmm_prepacked_weight_bytes")
    return out.value


def wqbmm_prepack_weight(w_packed, w_prepacked, K: int, N: int, G: int, stream=None) -> None:
    _check(load_library().wqbmm_prepack_weight(_ptr(w_packed), _ptr(w_prepacked), K, N, G, _stream(stream)),
           "wqbmm_prepack_weight")


def wqbmm_prepack_weight_nk(w_packed_nk, w_prepacked, K: int, N: int, G: int, stream=None) -> None:
    _check(load_library().wqbmm_prepack_weight_nk(_ptr(w_packed_nk), _ptr(w_prepacked), K, N, G, _stream(stream)),
           "wqbmm_prepack_weight_nk")


def wqbmm_workspace_bytes(M: int, K: int, N: int, G: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load_library().wqbmm_workspace_bytes(M, K, N, G, ctypes.byref(out)), "wqbmm_workspace_bytes")
    return out.value


def wqbmm_run(x, w_prepacked, antiquant_scale, y, M: int, K: int, N: int, G: int, workspace=None,
              workspace_bytes: int | None = None, stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().wqbmm_run(_ptr(x), _ptr(w_prepacked), _ptr(antiquant_scale), _ptr(y), M, K, N, G,
                                     _ptr(workspace), workspace_bytes, _stream(stream)), "wqbmm_run")


def wqbmm_run_ex(x, w_prepacked, antiquant_scale, zero_point, bias, y, M: int, K: int, N: int, G: int,
                 workspace=None, workspace_bytes: int | None = None, stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().wqbmm_run_ex(_ptr(x), _ptr(w_prepacked), _ptr(antiquant_scale), _ptr(zero_point),
                                        _ptr(bias), _ptr(y), M, K, N, G, _ptr(workspace), workspace_bytes,
                                        _stream(stream)), "wqbmm_run_ex")


def wqbmm_run_part(x, w_prepacked, antiquant_scale, zero_point, bias, y, M: int, K: int, N: int, G: int,
                   workspace=None, workspace_bytes: int | None = None, part: int = 0, stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().wqbmm_run_part(_ptr(x), _ptr(w_prepacked), _ptr(antiquant_scale), _ptr(zero_point),
                                          _ptr(bias), _ptr(y), M, K, N, G, _ptr(workspace), workspace_bytes, int(part),
                                          _stream(stream)), "wqbmm_run_part")


def wqbmm_run_batched(x, w_prepacked, antiquant_scale, zero_point, bias, y, batch: int, M: int, K: int, N: int,
                      G: int, x_batch_stride: int, y_batch_stride: int, workspace=None,
                      workspace_bytes: int | None = None, stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().wqbmm_run_batched(_ptr(x), _ptr(w_prepacked), _ptr(antiquant_scale), _ptr(zero_point),
                                             _ptr(bias), _ptr(y), batch, M, K, N, G, x_batch_stride, y_batch_stride,
                                             _ptr(workspace), workspace_bytes, _stream(stream)), "wqbmm_run_batched")


def wqbmm_prepacked_weight_bytes_w8(K: int, N: int, G: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load_library().wqbmm_prepacked_weight_bytes_w8(K, N, G, ctypes.byref(out)),
           "wqbmm_prepacked_weight_bytes_w8")
    return out.value


def wqbmm_prepack_weight_w8(w8, w_prepacked, K: int, N: int, G: int, stream=None) -> None:
    _check(load_library().wqbmm_prepack_weight_w8(_ptr(w8), _ptr(w_prepacked), K, N, G, _stream(stream)),
           "wqbmm_prepack_weight_w8")


def wqbmm_workspace_bytes_w8(M: int, K: int, N: int, G: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load_library().wqbmm_workspace_bytes_w8(M, K, N, G, ctypes.byref(out)), "wqbmm_workspace_bytes_w8")
    return out.value


def wqbmm_run_w8(x, w_prepacked, antiquant_scale, zero_point, bias, y, M: int, K: int, N: int, G: int,
                 workspace=None, workspace_bytes: int | None = None, stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().wqbmm_run_w8(_ptr(x), _ptr(w_prepacked), _ptr(antiquant_scale), _ptr(zero_point),
                                        _ptr(bias), _ptr(y), M, K, N, G, _ptr(workspace), workspace_bytes,
                                        _stream(stream)), "wqbmm_run_w8")


def wqbmm_run_static_scratch(x, w_prepacked, antiquant_scale, y, M: int, K: int, N: int, G: int,
                             stream=None) -> None:
    """wqbmm_run without a caller workspace: the library's fixed 2 MiB device scratch is used instead (for callers
    that cannot allocate device memory). Calls must not overlap on the GPU; the first call on a device looks up the
    scratch address and should come before any stream capture."""
    _check(load_library().wqbmm_run_static_scratch(_ptr(x), _ptr(w_prepacked), _ptr(antiquant_scale), _ptr(y), M, K,
                                                    N, G, _stream(stream)), "wqbmm_run_static_scratch")


def wqbmm_debug_unfold(x, M: int, K: int, G: int, planes, amax, stream=None) -> None:
    _check(load_library().wqbmm_debug_unfold(_ptr(x), M, K, G, _ptr(planes), _ptr(amax), _stream(stream)),
           "wqbmm_debug_unfold")


def wqbmm_debug_group_partials(x, w_prepacked, M: int, K: int, N: int, G: int, g: int, y123, workspace=None,
                               workspace_bytes: int | None = None, stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().wqbmm_debug_group_partials(_ptr(x), _ptr(w_prepacked), M, K, N, G, g, _ptr(y123),
                                                     _ptr(workspace), workspace_bytes, _stream(stream)),
           "wqbmm_debug_group_partials")


def wqbmm_read_device_status(clear: bool = False, stream=None) -> int:
    code = ctypes.c_int32(0)
    _check(load_library().wqbmm_read_device_status(ctypes.byref(code), int(bool(clear)), _stream(stream)),
           "wqbmm_read_device_status")
    return code.value


def wqbmm_debug_wait_timeout(limit_ns: int, stream=None) -> None:
    _check(load_library().wqbmm_debug_wait_timeout(limit_ns, _stream(stream)), "wqbmm_debug_wait_timeout")


# ---------------------------------------------------------------------------- allocation helpers (torch memory)

def prepack_weight(w_packed, K: int, N: int, G: int, stream=None):
    """uint8 [K/2, N] packed int4 on the GPU -> a new uint8 tensor in the prepacked tile layout."""
    import torch
    out = torch.empty(wqbmm_prepacked_weight_bytes(K, N, G), dtype=torch.uint8, device=w_packed.device)
    wqbmm_prepack_weight(w_packed, out, K, N, G, stream)
    return out


def prepack_weight_nk(w_packed_nk, K: int, N: int, G: int, stream=None):
    """uint8 [N, K/2] packed int4 (a weight stored transposed) on the GPU -> a new prepacked uint8 tensor."""
    import torch
    out = torch.empty(wqbmm_prepacked_weight_bytes(K, N, G), dtype=torch.uint8, device=w_packed_nk.device)
    wqbmm_prepack_weight_nk(w_packed_nk, out, K, N, G, stream)
    return out


def prepack_weight_w8(w8, K: int, N: int, G: int, stream=None):
    """int8 [K, N] weights on the GPU -> a new uint8 tensor of prepacked split (int4) tiles."""
    import torch
    out = torch.empty(wqbmm_prepacked_weight_bytes_w8(K, N, G), dtype=torch.uint8, device=w8.device)
    wqbmm_prepack_weight_w8(w8, out, K, N, G, stream)
    return out


def msd_matmul_w8(x, w_prepacked, antiquant_scale, G: int, y=None, workspace=None, stream=None, zero_point=None,
                  bias=None):
    """y [M, N] fp16 = MSD matmul of x [M, K] fp16 with prepacked int8 weights (prepack_weight_w8)."""
    import torch
    M, K = x.shape
    N = antiquant_scale.shape[1]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    if M == 0:
        wqbmm_workspace_bytes_w8(1, K, N, G)        # the library still checks K, N and G; no rows, nothing to run
        return y
    _check_operands(x, w_prepacked, antiquant_scale, zero_point, bias, y, (M, N), K, N, G, M,
                    wqbmm_prepacked_weight_bytes_w8(K, N, G))
    if workspace is None:
        workspace = torch.zeros(wqbmm_workspace_bytes_w8(M, K, N, G), dtype=torch.uint8, device=x.device)
    wqbmm_run_w8(x, w_prepacked, antiquant_scale, zero_point, bias, y, M, K, N, G, workspace, None, stream)
    return y


def _check_operands(x, w_prepacked, scale, zero_point, bias, y, y_shape, K: int, N: int, G: int, M: int,
                    w_bytes: int) -> None:
    """Shapes, dtypes, contiguity and devices of the tensors handed to the C ABI, which sees only raw pointers: a
    buffer that is too small or on another device would be read or written out of bounds by the kernels."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device())
    groups = K // G if G != K else 1
    named = [("x", x, torch.float16, None), ("y", y, torch.float16, tuple(y_shape)),
             ("antiquant_scale", scale, torch.float16, (groups, N)), ("w_prepacked", w_prepacked, None, None)]
    if zero_point is not None:
        named.append(("zero_point", zero_point, torch.float16, (groups, N)))
    if bias is not None:
        named.append(("bias", bias, torch.float16, (N,)))
    for name, t, dtype, shape in named:
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch tensor")
        if t.device != dev:
            raise ValueError(f"{name} is on {t.device}, the current CUDA device is {dev}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if dtype is not None and t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
        if shape is not None and tuple(t.shape) != shape:
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {shape}")
    if tuple(x.shape)[-1] != K:
        raise ValueError(f"x has {tuple(x.shape)[-1]} columns, expected K = {K}")
    if w_prepacked.numel() * w_prepacked.element_size() < w_bytes:
        raise ValueError(f"w_prepacked holds {w_prepacked.numel() * w_prepacked.element_size()} bytes, the "
                         f"prepacked layout of K = {K}, N = {N} needs {w_bytes}")


def allocate_workspace(M: int, K: int, N: int, G: int, device):
    """Zero-filled workspace for wqbmm_run (None when the shape needs none)."""
    import torch
    nbytes = wqbmm_workspace_bytes(M, K, N, G)
    if nbytes == 0:
        return None
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


def msd_matmul(x, w_prepacked, antiquant_scale, G: int, y=None, workspace=None, stream=None, zero_point=None,
               bias=None):
    """y [..., N] fp16 = MSD matmul of x [..., K] fp16 (any leading batch dimensions, contiguous) with prepacked int4
    weights and antiquant_scale [K/G, N] fp16 (G = K: per channel, [1, N]); optionally with zero points [K/G, N] fp16
    (weights (w - zp) * scale) and a bias [N] fp16."""
    import torch
    lead = tuple(x.shape[:-1])
    K = x.shape[-1]
    M = 1
    for d in lead:
        M *= d
    N = antiquant_scale.shape[1]
    if y is None:
        y = torch.empty(lead + (N,), dtype=torch.float16, device=x.device)
    if M == 0:
        wqbmm_workspace_bytes(1, K, N, G)           # the library still checks K, N and G; no rows, nothing to run
        return y
    _check_operands(x, w_prepacked, antiquant_scale, zero_point, bias, y, lead + (N,), K, N, G, M,
                    wqbmm_prepacked_weight_bytes(K, N, G))
    if workspace is None:
        workspace = allocate_workspace(M, K, N, G, x.device)
    if zero_point is None and bias is None:
        wqbmm_run(x, w_prepacked, antiquant_scale, y, M, K, N, G, workspace, None, stream)
    else:
        wqbmm_run_ex(x, w_prepacked, antiquant_scale, zero_point, bias, y, M, K, N, G, workspace, None, stream)
    return y
