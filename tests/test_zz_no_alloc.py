"""wqbmm_run_static_scratch: the allocation-free variant of wqbmm_run.

Some callers cannot allocate device memory: their memory belongs to another allocator (a framework's caching pool,
a plugin slot that receives only input and output buffers), so they have no workspace to hand to wqbmm_run. This
entry point uses a fixed device array inside the library instead. These tests call it through the C ABI and check
that it gives wqbmm_run's result (within the fp16 tolerance the parity tests use), on calls in a row, including a
change of shape in between (the array keeps the previous call's contents, so the counters must be cleared), and
that a shape needing more than the array holds is refused before anything runs.
"""
import numpy as np
import pytest

import weight_quantized_matmul_gb300 as wq
from weight_quantized_matmul_gb300 import build as wqbuild
from weight_quantized_matmul_gb300 import inputs as I

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def fp16_ulp(v):
    a = np.abs(np.asarray(v, dtype=np.float64))
    return 2.0 ** (np.floor(np.log2(np.maximum(a, 2.0 ** -14))) - 10)


def within_tolerance(got, ref):
    got = got.astype(np.float64)
    ref = ref.astype(np.float64)
    return np.abs(got - ref) <= 2e-3 * np.abs(ref).max() + fp16_ulp(ref)


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    wqbuild.build()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


# shapes whose split over K goes through the scratch (more K-slices than one thread-block cluster holds)
SHAPES = {
    "long_k_m1_k65536_n256": I.small_case(1, 65536, 256, 128, seed=11),
    "m3_k16384_n520_g64": I.small_case(3, 16384, 520, 64, seed=12),
}


def device_problem(name, dev):
    wl = SHAPES[name]
    x, wp, sc = I.make_inputs(wl)
    xd = torch.from_numpy(x).to(dev)
    sd = torch.from_numpy(sc).to(dev)
    w_pre = wq.prepack_weight(torch.from_numpy(wp).to(dev), wl.K, wl.N, wl.G)
    return wl, xd, w_pre, sd


def reference_run(wl, xd, w_pre, sd, dev):
    y = torch.empty((wl.M, wl.N), dtype=torch.float16, device=dev)
    ws = wq.allocate_workspace(wl.M, wl.K, wl.N, wl.G, dev)
    wq.wqbmm_run(xd, w_pre, sd, y, wl.M, wl.K, wl.N, wl.G, ws)
    return y.cpu().numpy()


@pytest.mark.parametrize("order", [("long_k_m1_k65536_n256", "long_k_m1_k65536_n256", "m3_k16384_n520_g64"),
                                   ("m3_k16384_n520_g64", "long_k_m1_k65536_n256", "m3_k16384_n520_g64")])
def test_static_scratch_matches_run_on_calls_in_a_row(dev, order):
    problems = {name: device_problem(name, dev) for name in set(order)}
    refs = {name: reference_run(*problems[name], dev) for name in problems}
    for name in order:
        wl, xd, w_pre, sd = problems[name]
        assert wq.wqbmm_workspace_bytes(wl.M, wl.K, wl.N, wl.G) > 0     # this shape does use scratch
        y = torch.full((wl.M, wl.N), float("nan"), dtype=torch.float16, device=dev)
        wq.wqbmm_run_static_scratch(xd, w_pre, sd, y, wl.M, wl.K, wl.N, wl.G)
        got = y.cpu().numpy()
        assert within_tolerance(got, refs[name]).all(), name
    torch.cuda.synchronize()
    assert wq.wqbmm_read_device_status() == 0


def test_static_scratch_refuses_shapes_beyond_its_size(dev):
    # 16 column tiles of 16 rows split over K 19 times: 19 x 16 x 2048 fp32 partial sums = 2.5 MB > 2 MiB
    M, K, N, G = 16, 4096, 2048, 128
    assert wq.wqbmm_workspace_bytes(M, K, N, G) > 2 * 1024 * 1024
    x = torch.zeros((M, K), dtype=torch.float16, device=dev)
    s = torch.zeros((K // G, N), dtype=torch.float16, device=dev)
    w_pre = torch.zeros(wq.wqbmm_prepacked_weight_bytes(K, N, G), dtype=torch.uint8, device=dev)
    y = torch.full((M, N), 3.0, dtype=torch.float16, device=dev)
    with pytest.raises(wq.WqbmmError) as e:
        wq.wqbmm_run_static_scratch(x, w_pre, s, y, M, K, N, G)
    assert e.value.status == wq.ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert (y == 3.0).all()
