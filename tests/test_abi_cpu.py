"""The C-ABI library builds for sm_103a, loads, exports every entry point include/wqbmm.h declares, and rejects bad
arguments before touching a device (status codes in the manner of the page "aclnnCalculateMatmulWeightSizeV2
接口详解", section on return values: null pointers, invalid parameters and platform errors are distinct codes).
None of these tests launches a kernel.
"""
import os
import re
import subprocess

import pytest

import weight_quantized_matmul_gb300 as wq
from weight_quantized_matmul_gb300 import build as wqbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "wqbmm.h")
A = 0x10000          # a 16-byte aligned fake device address: validation must reject before any use of it
MIS = 0x10008        # 8-byte aligned only


@pytest.fixture(scope="module")
def lib():
    wqbuild.build()
    return wq.load_library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^WQBMM_API\s+(?:const\s+)?\w+\s*\*?\s*(wqbmm_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_binding_symbols():
    assert declared_functions() == sorted(wq.SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", wq.library_path()], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\b(wqbmm_\w+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)
    # nothing but the C ABI leaks out of the library
    assert all(s.startswith("wqbmm_") for s in exported)


def test_build_targets_sm_103a_only():
    flags = " ".join(wqbuild.NVCC_FLAGS)
    assert flags.count("-gencode") == 1 and "arch=compute_103a,code=sm_103a" in flags


def test_status_strings(lib):
    for code in range(7):
        assert wq.wqbmm_status_string(code).startswith("WQBMM_")
    assert "UNKNOWN" in wq.wqbmm_status_string(99)


def test_prepacked_weight_bytes():
    assert wq.wqbmm_prepacked_weight_bytes(4096, 4096, 128) == 4096 * 4096 // 2
    assert wq.wqbmm_prepacked_weight_bytes(96, 1000, 32) == 8 * 1 * 8192     # padded to 128 x 128 tiles
    assert wq.wqbmm_prepacked_weight_bytes(8192, 28672, 64) == 8192 * 28672 // 2


def test_workspace_bytes():
    # M <= 2: int8 planes (3 bytes per element of x) + a float4 of constants per row and group
    assert wq.wqbmm_workspace_bytes(1, 4096, 4096, 128) == 3 * 4096 + 16 * 32
    assert wq.wqbmm_workspace_bytes(2, 65536, 256, 128) == 2 * 3 * 65536 + 2 * 16 * 512
    assert wq.wqbmm_workspace_bytes(1, 320, 136, 64) == 1280 + 256     # 3 x 384 and 5 x 16, each in 256-byte blocks
    # 3 <= M < 64: x unfolded once per 128 k into the tensor-core operand image (three planes of up to 16 rows:
    # 16, 32 or 48 rows x 128 bytes per row tile and k-block) plus 8 x 16 floats of constants per group. 8 column
    # tiles of 16 rows split over K into 8 slices that reduce inside a thread-block cluster need nothing more
    assert wq.wqbmm_workspace_bytes(16, 1024, 1024, 128) == 8 * 48 * 128 + 8 * 512
    # G = 32 (four groups per k-block): row tiles of at most 10 rows, so 16 rows are two tiles of 8 (MMA N = 32);
    # with G = 64 one tile of 16 (N = 48)
    assert wq.wqbmm_workspace_bytes(16, 1024, 1024, 32) == 2 * 8 * 32 * 128 + 2 * 32 * 512
    assert wq.wqbmm_workspace_bytes(16, 1024, 1024, 64) == 8 * 48 * 128 + 16 * 512
    # two column tiles and a long K: 160 slices (sized for up to 160 SMs, two CTAs each) reduce through the
    # workspace: 160 x 3 x 256 fp32 partial sums + one 256-byte block of counters after the unfolded x
    assert wq.wqbmm_workspace_bytes(3, 65536, 256, 128) == 512 * 16 * 128 + 512 * 512 + 160 * 3 * 256 * 4 + 256
    assert wq.wqbmm_workspace_bytes(40, 1024, 28672, 128) == 3 * 8 * 48 * 128 + 3 * 8 * 512


def test_w8_sizes():
    # the split weights have 2K rows of int4: K * N bytes, padded to whole tiles
    assert wq.wqbmm_prepacked_weight_bytes_w8(4096, 4096, 128) == 4096 * 4096
    assert wq.wqbmm_prepacked_weight_bytes_w8(96, 1000, 32) == 8 * 2 * 8192
    # workspace: the int4 problem's (M, 2K) plus x repeated [M, 2K] and the split scales and zero points
    M, K, N, G = 1, 4096, 4096, 128
    assert wq.wqbmm_workspace_bytes_w8(M, K, N, G) == (wq.wqbmm_workspace_bytes(M, 2 * K, N, G) + _a256(M * 2 * K * 2)
                                                       + 2 * _a256(2 * (K // G) * N * 2))


def _a256(v):
    return (v + 255) // 256 * 256


def test_workspace_bytes_per_channel():
    # G = K: the kernels work in 128-k sub-groups with each row's A_max; the decode path adds the row maxima,
    # the others also the scale and zero-point rows repeated per sub-group
    assert wq.wqbmm_workspace_bytes(1, 4096, 4096, 4096) == 3 * 4096 + 16 * 32 + _a256(4)
    assert wq.wqbmm_workspace_bytes(8, 4096, 11008, 4096) == (32 * 32 * 128 + 32 * 512 + _a256(8 * 4) +
                                                               2 * _a256(32 * 11008 * 2))
    assert wq.wqbmm_workspace_bytes(256, 1024, 392, 1024) == (3 * 256 * 1024 + 16 * 256 * 8 + _a256(256 * 4) +
                                                                2 * _a256(8 * 392 * 2))
    # K not a multiple of 128: sub-groups of 32
    assert wq.wqbmm_workspace_bytes(2, 352, 136, 352) == _a256(2 * 3 * 384) + _a256(2 * 11 * 16) + _a256(8)
    # G = K = 64 is an ordinary group (same arithmetic): no per-channel extras
    assert wq.wqbmm_workspace_bytes(1, 64, 128, 64) == 256 * 2 + 256
    # M >= 64: x unfolded once into three planes of 128-row tiles (3 bytes per element of x, rows padded to 128)
    # plus 16 bytes of combine constants per padded row and group
    assert wq.wqbmm_workspace_bytes(2048, 8192, 28672, 64) == 3 * 2048 * 8192 + 16 * 2048 * 128
    assert wq.wqbmm_workspace_bytes(128, 5120, 13824, 128) == 3 * 128 * 5120 + 16 * 128 * 40
    assert wq.wqbmm_workspace_bytes(64, 320, 136, 64) == 3 * 128 * 384 + 16 * 128 * 5
    # 63 rows is still the small-M path: four row tiles of 16, enough column tiles, no split
    assert wq.wqbmm_workspace_bytes(63, 4096, 28672, 64) == 4 * 32 * 48 * 128 + 4 * 64 * 512


# (entry, args, expected status) — table-driven error paths
NULLPTR, INVALID = wq.ERR_NULLPTR, wq.ERR_INVALID
CASES = [
    ("size_null", lambda L: L.wqbmm_prepacked_weight_bytes(128, 128, 128, None), NULLPTR),
    ("size_bad_group", lambda L: L.wqbmm_prepacked_weight_bytes(128, 128, 48, _sz()), INVALID),
    ("size_k_not_multiple_of_group", lambda L: L.wqbmm_prepacked_weight_bytes(96, 128, 64, _sz()), INVALID),
    ("size_n_not_multiple_of_8", lambda L: L.wqbmm_prepacked_weight_bytes(128, 12, 128, _sz()), INVALID),
    ("size_zero_k", lambda L: L.wqbmm_prepacked_weight_bytes(0, 128, 128, _sz()), INVALID),
    ("size_negative_n", lambda L: L.wqbmm_prepacked_weight_bytes(128, -8, 128, _sz()), INVALID),
    ("size_k_too_large", lambda L: L.wqbmm_prepacked_weight_bytes(1 << 31, 8, 128, _sz()), INVALID),
    ("ws_null", lambda L: L.wqbmm_workspace_bytes(1, 128, 128, 128, None), NULLPTR),
    ("ws_zero_m", lambda L: L.wqbmm_workspace_bytes(0, 128, 128, 128, _sz()), INVALID),
    ("prepack_null_src", lambda L: L.wqbmm_prepack_weight(None, A, 128, 128, 128, None), NULLPTR),
    ("prepack_null_dst", lambda L: L.wqbmm_prepack_weight(A, None, 128, 128, 128, None), NULLPTR),
    ("prepack_misaligned_dst", lambda L: L.wqbmm_prepack_weight(A, MIS, 128, 128, 128, None), INVALID),
    ("prepack_bad_group", lambda L: L.wqbmm_prepack_weight(A, A, 128, 128, 16, None), INVALID),
    ("prepack_nk_null_src", lambda L: L.wqbmm_prepack_weight_nk(None, A, 128, 128, 128, None), NULLPTR),
    ("prepack_nk_misaligned_dst", lambda L: L.wqbmm_prepack_weight_nk(A, MIS, 128, 128, 128, None), INVALID),
    ("prepack_nk_bad_shape", lambda L: L.wqbmm_prepack_weight_nk(A, A, 96, 128, 64, None), INVALID),
    ("run_null_x", lambda L: L.wqbmm_run(None, A, A, A, 1, 128, 128, 128, A, 1 << 20, None), NULLPTR),
    ("run_null_w", lambda L: L.wqbmm_run(A, None, A, A, 1, 128, 128, 128, A, 1 << 20, None), NULLPTR),
    ("run_null_scale", lambda L: L.wqbmm_run(A, A, None, A, 1, 128, 128, 128, A, 1 << 20, None), NULLPTR),
    ("run_null_y", lambda L: L.wqbmm_run(A, A, A, None, 1, 128, 128, 128, A, 1 << 20, None), NULLPTR),
    ("run_null_workspace_needed", lambda L: L.wqbmm_run(A, A, A, A, 1, 65536, 256, 128, None, 0, None), NULLPTR),
    ("run_zero_m", lambda L: L.wqbmm_run(A, A, A, A, 0, 128, 128, 128, A, 1 << 20, None), INVALID),
    ("run_negative_k", lambda L: L.wqbmm_run(A, A, A, A, 1, -128, 128, 128, A, 1 << 20, None), INVALID),
    ("run_k_not_multiple_of_group", lambda L: L.wqbmm_run(A, A, A, A, 1, 160, 128, 128, A, 1 << 20, None),
     INVALID),
    ("run_group_not_supported", lambda L: L.wqbmm_run(A, A, A, A, 1, 192, 128, 96, A, 1 << 20, None), INVALID),
    ("run_n_ragged_by_4", lambda L: L.wqbmm_run(A, A, A, A, 1, 128, 132, 128, A, 1 << 20, None), INVALID),
    ("run_m_too_large", lambda L: L.wqbmm_run(A, A, A, A, 1 << 31, 128, 128, 128, A, 1 << 20, None), INVALID),
    ("run_misaligned_x", lambda L: L.wqbmm_run(MIS, A, A, A, 1, 128, 128, 128, A, 1 << 20, None), INVALID),
    ("run_misaligned_y", lambda L: L.wqbmm_run(A, A, A, MIS, 1, 128, 128, 128, A, 1 << 20, None), INVALID),
    ("run_misaligned_scale", lambda L: L.wqbmm_run(A, A, MIS, A, 1, 128, 128, 128, A, 1 << 20, None), INVALID),
    ("run_misaligned_weights", lambda L: L.wqbmm_run(A, MIS, A, A, 1, 128, 128, 128, A, 1 << 20, None), INVALID),
    ("run_misaligned_workspace", lambda L: L.wqbmm_run(A, A, A, A, 1, 65536, 256, 128, MIS, 1 << 20, None),
     INVALID),
    ("run_ex_null_x", lambda L: L.wqbmm_run_ex(None, A, A, A, A, A, 1, 128, 128, 128, A, 1 << 20, None), NULLPTR),
    ("run_ex_null_scale", lambda L: L.wqbmm_run_ex(A, A, None, A, A, A, 1, 128, 128, 128, A, 1 << 20, None),
     NULLPTR),
    ("run_ex_null_y", lambda L: L.wqbmm_run_ex(A, A, A, A, A, None, 1, 128, 128, 128, A, 1 << 20, None), NULLPTR),
    ("run_ex_misaligned_zero_point",
     lambda L: L.wqbmm_run_ex(A, A, A, MIS, None, A, 1, 128, 128, 128, A, 1 << 20, None), INVALID),
    ("run_ex_misaligned_bias",
     lambda L: L.wqbmm_run_ex(A, A, A, None, MIS, A, 200, 128, 128, 128, A, 1 << 20, None), INVALID),
    ("run_ex_bad_group", lambda L: L.wqbmm_run_ex(A, A, A, A, A, A, 8, 128, 128, 16, A, 1 << 20, None), INVALID),
    ("batched_zero_batch",
     lambda L: L.wqbmm_run_batched(A, A, A, None, None, A, 0, 2, 128, 128, 128, 256, 256, A, 1 << 20, None), INVALID),
    ("batched_x_stride_too_small",
     lambda L: L.wqbmm_run_batched(A, A, A, None, None, A, 2, 2, 128, 128, 128, 200, 256, A, 1 << 20, None), INVALID),
    ("batched_y_stride_unaligned",
     lambda L: L.wqbmm_run_batched(A, A, A, None, None, A, 2, 2, 128, 128, 128, 256, 260, A, 1 << 20, None), INVALID),
    ("batched_null_x",
     lambda L: L.wqbmm_run_batched(None, A, A, None, None, A, 2, 2, 128, 128, 128, 256, 256, A, 1 << 20, None),
     NULLPTR),
    ("batched_bad_group",
     lambda L: L.wqbmm_run_batched(A, A, A, None, None, A, 2, 2, 192, 128, 96, 512, 512, A, 1 << 20, None), INVALID),
    ("w8_size_per_channel_rejected", lambda L: L.wqbmm_prepacked_weight_bytes_w8(256, 128, 256, _sz()), INVALID),
    ("w8_prepack_null", lambda L: L.wqbmm_prepack_weight_w8(None, A, 256, 128, 128, None), NULLPTR),
    ("w8_prepack_misaligned", lambda L: L.wqbmm_prepack_weight_w8(A, MIS, 256, 128, 128, None), INVALID),
    ("w8_run_null_workspace",
     lambda L: L.wqbmm_run_w8(A, A, A, None, None, A, 1, 256, 128, 128, None, 0, None), NULLPTR),
    ("w8_run_bad_group", lambda L: L.wqbmm_run_w8(A, A, A, None, None, A, 1, 256, 128, 256, A, 1 << 20, None),
     INVALID),
    ("w8_ws_null", lambda L: L.wqbmm_workspace_bytes_w8(1, 256, 128, 128, None), NULLPTR),
    ("run_per_channel_k_not_multiple_of_32",
     lambda L: L.wqbmm_run(A, A, A, A, 1, 100, 128, 100, A, 1 << 20, None), INVALID),
    ("run_group_larger_than_128_not_k", lambda L: L.wqbmm_run(A, A, A, A, 1, 512, 128, 256, A, 1 << 20, None),
     INVALID),
    ("partials_per_channel_not_exposed",
     lambda L: L.wqbmm_debug_group_partials(A, A, 1, 256, 128, 256, 0, A, A, 1 << 20, None), INVALID),
    ("run_ex_null_workspace_needed",
     lambda L: L.wqbmm_run_ex(A, A, A, A, A, A, 1, 65536, 256, 128, None, 0, None), NULLPTR),
    ("unfold_null_planes", lambda L: L.wqbmm_debug_unfold(A, 1, 128, 128, None, A, None), NULLPTR),
    ("unfold_bad_group", lambda L: L.wqbmm_debug_unfold(A, 1, 128, 100, A, A, None), INVALID),
    ("partials_group_out_of_range",
     lambda L: L.wqbmm_debug_group_partials(A, A, 1, 256, 128, 128, 2, A, None, 0, None), INVALID),
    ("partials_negative_group",
     lambda L: L.wqbmm_debug_group_partials(A, A, 1, 256, 128, 128, -1, A, None, 0, None), INVALID),
    ("partials_large_m_needs_workspace",
     lambda L: L.wqbmm_debug_group_partials(A, A, 64, 256, 128, 128, 0, A, None, 0, None), NULLPTR),
    ("partials_large_m_workspace_too_small",
     lambda L: L.wqbmm_debug_group_partials(A, A, 64, 256, 128, 128, 0, A, A, 1024, None), INVALID),
    ("static_scratch_null_y", lambda L: L.wqbmm_run_static_scratch(A, A, A, None, 1, 128, 128, 128, None),
     NULLPTR),
    ("static_scratch_misaligned_x", lambda L: L.wqbmm_run_static_scratch(MIS, A, A, A, 1, 128, 128, 128, None),
     INVALID),
    ("static_scratch_bad_group", lambda L: L.wqbmm_run_static_scratch(A, A, A, A, 1, 128, 128, 96, None), INVALID),
    ("run_part_bad_part",
     lambda L: L.wqbmm_run_part(A, A, A, None, None, A, 1, 128, 128, 128, A, 1 << 20, 3, None), INVALID),
    ("run_part_null_y",
     lambda L: L.wqbmm_run_part(A, A, A, None, None, None, 1, 128, 128, 128, A, 1 << 20, 2, None), NULLPTR),
    ("status_null", lambda L: L.wqbmm_read_device_status(None, 0, None), NULLPTR),
    ("timeout_limit_too_small", lambda L: L.wqbmm_debug_wait_timeout(10, None), INVALID),
    ("timeout_limit_too_large", lambda L: L.wqbmm_debug_wait_timeout(10 ** 10, None), INVALID),
]


def _sz():
    import ctypes
    return ctypes.byref(ctypes.c_size_t(0))


@pytest.mark.parametrize("name,call,want", CASES, ids=[c[0] for c in CASES])
def test_rejected_before_any_device_work(lib, name, call, want):
    assert call(lib) == want


def test_no_device_is_a_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    # valid arguments, but no GPU: the device check fails with a CUDA error and nothing is launched
    assert lib.wqbmm_run(A, A, A, A, 16, 8192, 28672, 64, A, 1 << 30, None) == wq.ERR_CUDA
    assert lib.wqbmm_run(A, A, A, A, 2048, 8192, 28672, 64, A, 1 << 30, None) == wq.ERR_CUDA
    assert lib.wqbmm_run_ex(A, A, A, A, A, A, 8, 4096, 11008, 128, A, 1 << 30, None) == wq.ERR_CUDA
    assert lib.wqbmm_run_ex(A, A, A, None, None, A, 1, 4096, 4096, 128, A, 1 << 30, None) == wq.ERR_CUDA
    assert lib.wqbmm_run_batched(A, A, A, None, None, A, 4, 2, 4096, 4096, 128, 8192, 8192, A, 1 << 30,
                                 None) == wq.ERR_CUDA
    assert lib.wqbmm_run_w8(A, A, A, None, None, A, 8, 4096, 11008, 128, A, 1 << 30, None) == wq.ERR_CUDA
    assert lib.wqbmm_prepack_weight_w8(A, A, 4096, 4096, 128, None) == wq.ERR_CUDA
    assert lib.wqbmm_run_batched(A, A, A, None, None, A, 4, 2, 4096, 4096, 128, 9216, 8192, A, 1 << 30,
                                 None) == wq.ERR_CUDA


def test_empty_batch_returns_an_empty_product(lib):
    # no rows: nothing to compute, y keeps the batch dimensions; the library still validates K, N and G
    import torch
    K, N, G = 512, 264, 128
    w = torch.empty(0, dtype=torch.uint8)
    s = torch.empty((K // G, N), dtype=torch.float16)
    for shape in [(0, K), (3, 0, K)]:
        y = wq.msd_matmul(torch.empty(shape, dtype=torch.float16), w, s, G)
        assert tuple(y.shape) == shape[:-1] + (N,) and y.dtype == torch.float16
    y8 = wq.msd_matmul_w8(torch.empty((0, K), dtype=torch.float16), w, s, G)
    assert tuple(y8.shape) == (0, N)
    with pytest.raises(Exception):
        wq.msd_matmul(torch.empty((0, K), dtype=torch.float16), w, torch.empty((K // 48, N)), 48)   # G not allowed
    with pytest.raises(Exception):
        wq.msd_matmul(torch.empty((0, K), dtype=torch.float16), w, torch.empty((K // G, 260)), G)   # N % 8 != 0
