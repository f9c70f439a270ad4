"""wqbmm_run_static_scratch: the allocation-free variant of wqbmm_run.

Some callers cannot allocate device memory: their memory belongs to another allocator (a framework's caching pool,
a plugin slot that receives only input and output buffers), so they have no workspace to hand to wqbmm_run. This
entry point uses a fixed device array inside the library instead. These tests call it through the C ABI and check,
on calls in a row (the array keeps each call's contents, so every call must rewrite what it reads):
  - that it gives wqbmm_run's result and the oracle's (within the fp16 tolerance the parity tests use), on every
    kernel path: decode rows, the small-M tensor-core kernel with its split over K reduced through the scratch, the
    large-M pre-pass and tiles, and per-channel scales, whose workspaces lay out the same array differently;
  - that a warmed-up call takes no device memory (the free memory the driver reports does not move);
  - that a shape needing more than the array holds is refused before anything runs.
"""
import numpy as np
import pytest

import oracle
import tolerance as T
import weight_quantized_matmul_gb300 as wq
from weight_quantized_matmul_gb300 import build as wqbuild
from weight_quantized_matmul_gb300 import inputs as I

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

SCRATCH_BYTES = 2 * 1024 * 1024


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    wqbuild.build()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


SHAPES = {
    "decode_m1_k4096_n4096": I.small_case(1, 4096, 4096, 128, seed=10),
    "long_k_m1_k65536_n256": I.small_case(1, 65536, 256, 128, seed=11),     # decode path, many passes
    "m3_k16384_n520_g64": I.small_case(3, 16384, 520, 64, seed=12),         # split over K through the scratch
    "large_m64_k1024_n1024": I.small_case(64, 1024, 1024, 128, seed=13),    # unfold pre-pass and 128-row tiles
    "per_channel_m8_k1024_n1024": I.small_case(8, 1024, 1024, 1024, seed=14),
}


def device_problem(name, dev):
    wl = SHAPES[name]
    x, wp, sc = I.make_inputs(wl)
    xd = torch.from_numpy(x).to(dev)
    sd = torch.from_numpy(sc).to(dev)
    w_pre = wq.prepack_weight(torch.from_numpy(wp).to(dev), wl.K, wl.N, wl.G)
    ref_d = oracle.msd_matmul(x, wp, sc, wl.G, mode=oracle.MODE_D)
    ref_f = oracle.msd_matmul(x, wp, sc, wl.G, mode=oracle.MODE_F)
    return wl, xd, w_pre, sd, ref_d, ref_f


def workspace_run(wl, xd, w_pre, sd, dev):
    y = torch.empty((wl.M, wl.N), dtype=torch.float16, device=dev)
    ws = wq.allocate_workspace(wl.M, wl.K, wl.N, wl.G, dev)
    wq.wqbmm_run(xd, w_pre, sd, y, wl.M, wl.K, wl.N, wl.G, ws)
    return y.cpu().numpy()


ORDERS = [
    ("decode_m1_k4096_n4096", "m3_k16384_n520_g64", "large_m64_k1024_n1024", "per_channel_m8_k1024_n1024",
     "long_k_m1_k65536_n256", "large_m64_k1024_n1024"),
    ("large_m64_k1024_n1024", "large_m64_k1024_n1024", "m3_k16384_n520_g64", "m3_k16384_n520_g64",
     "per_channel_m8_k1024_n1024", "decode_m1_k4096_n4096"),
]


@pytest.mark.parametrize("order", ORDERS)
def test_static_scratch_matches_run_and_oracle_on_calls_in_a_row(dev, order):
    problems = {name: device_problem(name, dev) for name in set(order)}
    runs = {name: workspace_run(*problems[name][:4], dev) for name in problems}
    for name in order:
        wl, xd, w_pre, sd, ref_d, ref_f = problems[name]
        assert 0 < wq.wqbmm_workspace_bytes(wl.M, wl.K, wl.N, wl.G) <= SCRATCH_BYTES   # the scratch is used
        y = torch.full((wl.M, wl.N), float("nan"), dtype=torch.float16, device=dev)
        wq.wqbmm_run_static_scratch(xd, w_pre, sd, y, wl.M, wl.K, wl.N, wl.G)
        got = y.cpu().numpy()
        T.assert_within_tolerance(got, runs[name].astype(np.float64), f"{name} against wqbmm_run")
        T.assert_matches(got, ref_d, ref_f, f"{name} against the oracle")
    torch.cuda.synchronize()
    assert wq.wqbmm_read_device_status() == 0


def test_static_scratch_takes_no_device_memory(dev):
    wl, xd, w_pre, sd, _, _ = device_problem("m3_k16384_n520_g64", dev)
    y = torch.empty((wl.M, wl.N), dtype=torch.float16, device=dev)
    wq.wqbmm_run_static_scratch(xd, w_pre, sd, y, wl.M, wl.K, wl.N, wl.G)        # warm-up: modules loaded
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        wq.wqbmm_run_static_scratch(xd, w_pre, sd, y, wl.M, wl.K, wl.N, wl.G)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before


def test_static_scratch_refuses_shapes_beyond_its_size(dev):
    # 16 column tiles of 16 rows split over K 19 times: 19 x 16 x 2048 fp32 partial sums = 2.5 MB > 2 MiB
    M, K, N, G = 16, 4096, 2048, 128
    assert wq.wqbmm_workspace_bytes(M, K, N, G) > SCRATCH_BYTES
    x = torch.zeros((M, K), dtype=torch.float16, device=dev)
    s = torch.zeros((K // G, N), dtype=torch.float16, device=dev)
    w_pre = torch.zeros(wq.wqbmm_prepacked_weight_bytes(K, N, G), dtype=torch.uint8, device=dev)
    y = torch.full((M, N), 3.0, dtype=torch.float16, device=dev)
    with pytest.raises(wq.WqbmmError) as e:
        wq.wqbmm_run_static_scratch(x, w_pre, s, y, M, K, N, G)
    assert e.value.status == wq.ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert (y == 3.0).all()
