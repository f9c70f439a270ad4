"""Parity of the CUDA path with the CPU oracle, through the C ABI, on a GB300.

Bars (method: WeightQuantBatchMatmulExperiment page, section 4.1):
  - prepacked weights: byte-exact against the documented tile layout;
  - steps 1-8 (A_max and the three planes, wqbmm_debug_unfold): bit-exact against the oracle's binary32 unfold;
  - step 9 (per-group integer Y1..Y3 from the tensor-core path, wqbmm_debug_group_partials): bit-exact;
  - steps 1-11 (wqbmm_run, fp16 y): |y - y_ref| <= 2e-3 * max|y_ref| + 1 fp16 ulp(y_ref) against the oracle in
    binary64 (and in binary32 unfold), element by element; at full workload sizes on seeded sampled rows; and the
    tight bar of tests/tolerance.py (the binary32-unfold oracle rounded to fp16, within 0.6 ulp, on every output
    that is not small), which sees an error in any one combine constant.
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


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    wqbuild.build()
    torch.cuda.set_device(0)
    wq.wqbmm_read_device_status(clear=True)
    return torch.device("cuda:0")


@pytest.fixture(autouse=True)
def device_status_clean(dev):
    yield
    torch.cuda.synchronize()
    assert wq.wqbmm_read_device_status() == 0


def to_dev(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def gpu_run(x, wp, sc, G, dev, M=None):
    M, K = x.shape
    N = sc.shape[1]
    xd, wd, sd = to_dev(x, dev), to_dev(wp, dev), to_dev(sc, dev)
    w_pre = wq.prepack_weight(wd, K, N, G)
    y = wq.msd_matmul(xd, w_pre, sd, G)
    return y.cpu().numpy()


def prepack_layout(wp, K, N):
    """The tile layout documented for wqbmm_prepacked_weight_bytes, restated with numpy."""
    nt, kb = -(-N // 128), -(-K // 128)
    padded = np.zeros((kb * 64, nt * 128), dtype=np.uint8)
    padded[:K // 2, :N] = wp
    padded ^= 0x88
    u = np.stack([padded & 0xF, padded >> 4], axis=1).reshape(kb * 128, nt * 128)      # u[k, n] = w + 8
    u = u.reshape(kb, 16, 2, 4, nt, 128)                                               # k = 128 kb + 8q + 4h + b
    byte = u[:, :, 0] | (u[:, :, 1] << 4)                                              # [kb, q, b, nt, 128]
    return byte.reshape(kb, 64, nt, 128).transpose(2, 0, 3, 1).reshape(-1)


# ------------------------------------------------------------------------------------------- prepack

@pytest.mark.parametrize("K,N,G", [(128, 128, 128), (4096, 4096, 128), (96, 1000, 32), (640, 264, 64)])
def test_prepack_matches_documented_layout(dev, K, N, G):
    wp = I.make_w_packed(I.small_case(1, K, N, G, seed=K + N))
    got = wq.prepack_weight(to_dev(wp, dev), K, N, G).cpu().numpy()
    np.testing.assert_array_equal(got, prepack_layout(wp, K, N))


def pack_int4_nk(w_packed_kn, K, N):
    """The [N, K/2] packing of the same weights (two k per byte, low nibble first), from their [K/2, N] packing."""
    w = oracle.decode_int4(w_packed_kn, K, N)                       # [K, N] int8
    u = (w.T.astype(np.int16) & 0xF).astype(np.uint8)               # [N, K] nibbles
    return np.ascontiguousarray(u[:, 0::2] | (u[:, 1::2] << 4))


@pytest.mark.parametrize("K,N,G", [(128, 128, 128), (640, 264, 64), (96, 1000, 32), (4096, 4096, 128)])
def test_prepack_of_transposed_weights_matches(dev, K, N, G):
    wp = I.make_w_packed(I.small_case(1, K, N, G, seed=K + 3 * N))
    nk = pack_int4_nk(wp, K, N)
    assert nk.shape == (N, K // 2)
    a = wq.prepack_weight(to_dev(wp, dev), K, N, G).cpu().numpy()
    b = wq.prepack_weight_nk(to_dev(nk, dev), K, N, G).cpu().numpy()
    np.testing.assert_array_equal(a, b)


NK_CASES = [
    # M, K, N, G: every kernel path, ragged N, K past 8192
    (1, 4096, 520, 128),            # decode kernel
    (2, 8320, 264, 64),             # decode kernel, K > 8192, ragged last CTA
    (3, 512, 1000, 32),             # small-M tensor-core kernel
    (16, 1024, 392, 64),            # small-M, cluster-reduced split-K
    (3, 16384, 136, 128),           # small-M, split-K through the workspace
    (64, 640, 264, 128),            # large-M
    (200, 1280, 136, 32),
]


@pytest.mark.parametrize("M,K,N,G", NK_CASES)
def test_transposed_weights_match_oracle(dev, M, K, N, G):
    """Weights given as [N, K/2] (the operator's transpose option for the weight, page 2 section 5.4), prepacked by
    wqbmm_prepack_weight_nk, then wqbmm_run and wqbmm_run_ex (fractional zero points and a bias): against the oracle,
    which reads the same weights in their [K/2, N] packing."""
    wl = I.small_case(M, K, N, G, seed=13 * M + K + N, x_dist="t3_clip60" if M % 2 else "normal")
    x, wp, sc = I.make_inputs(wl)
    zp, bias = I.make_zero_point(wl, "frac"), I.make_bias(wl)
    w_pre = wq.prepack_weight_nk(to_dev(pack_int4_nk(wp, K, N), dev), K, N, G)
    xd, sd = to_dev(x, dev), to_dev(sc, dev)
    ws = wq.allocate_workspace(M, K, N, G, dev)
    y = torch.empty((M, N), dtype=torch.float16, device=dev)
    wq.wqbmm_run(xd, w_pre, sd, y, M, K, N, G, ws)
    T.assert_matches(y.cpu().numpy(), oracle.msd_matmul(x, wp, sc, G, mode=oracle.MODE_D),
                     oracle.msd_matmul(x, wp, sc, G, mode=oracle.MODE_F), "transposed weights")
    y_ex = torch.empty((M, N), dtype=torch.float16, device=dev)
    wq.wqbmm_run_ex(xd, w_pre, sd, to_dev(zp, dev), to_dev(bias, dev), y_ex, M, K, N, G, ws)
    T.assert_matches(y_ex.cpu().numpy(),
                     oracle.msd_matmul_ex(x, wp, sc, G, zero_point=zp, bias=bias, mode=oracle.MODE_D),
                     oracle.msd_matmul_ex(x, wp, sc, G, zero_point=zp, bias=bias, mode=oracle.MODE_F),
                     "transposed weights, zero points and bias")


def test_binding_rejects_mismatched_tensors(dev):
    """The binding checks what the C ABI cannot see behind its raw pointers (shapes, dtypes, contiguity, devices,
    sizes) before anything is launched; the output is left untouched."""
    M, K, N, G = 4, 512, 264, 128
    x, wp, sc = I.make_inputs(I.small_case(M, K, N, G, seed=6))
    xd, sd = to_dev(x, dev), to_dev(sc, dev)
    w_pre = wq.prepack_weight(to_dev(wp, dev), K, N, G)
    y = torch.full((M, N), 5.0, dtype=torch.float16, device=dev)
    bad = [
        dict(y=torch.empty((M, N - 8), dtype=torch.float16, device=dev)),          # y too narrow
        dict(y=torch.empty((M, N), dtype=torch.float32, device=dev)),              # y of another dtype
        dict(antiquant_scale=sd[:2]),                                              # too few scale rows
        dict(antiquant_scale=torch.empty((N, K // G), dtype=torch.float16, device=dev).t()),   # not contiguous
        dict(x=xd.float()),                                                        # x of another dtype
        dict(w_prepacked=w_pre[:-16]),                                             # prepacked weights too short
        dict(zero_point=torch.zeros((K // G, N - 8), dtype=torch.float16, device=dev)),
        dict(bias=torch.zeros(N, dtype=torch.float16)),                            # bias on the host
    ]
    for kw in bad:
        args = dict(x=xd, w_prepacked=w_pre, antiquant_scale=sd, y=y)
        args.update(kw)
        with pytest.raises((ValueError, TypeError)):
            wq.msd_matmul(args.pop("x"), args.pop("w_prepacked"), args.pop("antiquant_scale"), G, **args)
    torch.cuda.synchronize()
    assert (y == 5.0).all()


# ------------------------------------------------------------------------------------------- steps 1-8

def special_x():
    """Rows that stress the unfold: ties in binary32, zero groups, subnormals, the fp16 extremes, -0."""
    rows = []
    r = np.zeros(128, dtype=np.float16)
    r[0], r[1] = 0.53125, 0.03857421875                # binary32 tie tmp3 = 2.5 (half-even -> 2)
    r[32], r[33] = 0.52294921875, 0.04107666015625     # tie tmp3 = -2.5
    rows.append(r)
    rows.append(np.zeros(128, dtype=np.float16))                       # all-zero groups
    r = np.full(128, -0.0, dtype=np.float16)
    r[5] = 5.960464477539063e-08                                       # smallest subnormal
    r[70] = -6.103515625e-05
    rows.append(r)
    r = I.fp16(np.linspace(-65504, 65504, 128))
    rows.append(r)
    allv = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
    fin = allv[np.isfinite(allv)]
    rng = fin[(I.raw_u64(99, 1, 0, 128 * 8) % np.uint64(fin.size)).astype(np.int64)].reshape(8, 128)
    rows.extend(list(rng))
    return np.stack(rows).astype(np.float16)


@pytest.mark.parametrize("G", [32, 64, 128])
@pytest.mark.parametrize("dist", ["normal", "t3_clip60", "normal_cols20", "uniform3"])
def test_unfold_bit_exact(dev, G, dist):
    x = I.make_x(I.small_case(37, 1024, 8, G, seed=G, x_dist=dist, x_sigma=3.0 if dist == "uniform3" else 1.0))
    M, K = x.shape
    planes = torch.empty((3, M, K), dtype=torch.int8, device=dev)
    amax = torch.empty((M, K // G), dtype=torch.float32, device=dev)
    wq.wqbmm_debug_unfold(to_dev(x, dev), M, K, G, planes, amax)
    p_ref, a_ref = oracle.unfold(x, G, oracle.MODE_F)
    np.testing.assert_array_equal(planes.cpu().numpy(), p_ref)
    np.testing.assert_array_equal(amax.cpu().numpy(), a_ref.astype(np.float32))


@pytest.mark.parametrize("G", [32, 64, 128])
def test_unfold_bit_exact_special_values(dev, G):
    x = special_x()
    M, K = x.shape
    planes = torch.empty((3, M, K), dtype=torch.int8, device=dev)
    amax = torch.empty((M, K // G), dtype=torch.float32, device=dev)
    wq.wqbmm_debug_unfold(to_dev(x, dev), M, K, G, planes, amax)
    p_ref, a_ref = oracle.unfold(x, G, oracle.MODE_F)
    np.testing.assert_array_equal(planes.cpu().numpy(), p_ref)
    np.testing.assert_array_equal(amax.cpu().numpy(), a_ref.astype(np.float32))


def test_unfold_bit_exact_every_fp16_value(dev):
    """Every finite fp16 x against 64 values of A_max (each group holds A_max and 127 values with |x| <= A_max),
    bit-exact against the oracle's binary32 unfold: the quotient step is exact over the whole domain."""
    allv = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
    fin = allv[np.isfinite(allv)]
    pos = np.sort(fin[fin > 0].astype(np.float64))
    pick = np.unique(np.concatenate([pos[np.linspace(0, pos.size - 1, 60).astype(int)],
                                     [5.960464477539063e-08, 6.103515625e-05, 1.0, 65504.0]]))[:64]
    G, K = 128, 65536
    rows = []
    for a in pick:
        vals = fin[np.abs(fin.astype(np.float64)) <= a]
        reps = -(-(K // G * (G - 1)) // vals.size)
        body = np.tile(vals, reps)[:K // G * (G - 1)].reshape(K // G, G - 1)
        rows.append(np.concatenate([np.full((K // G, 1), a, dtype=np.float16), body], axis=1).reshape(-1))
    x = np.stack(rows).astype(np.float16)
    M = x.shape[0]
    planes = torch.empty((3, M, K), dtype=torch.int8, device=dev)
    amax = torch.empty((M, K // G), dtype=torch.float32, device=dev)
    wq.wqbmm_debug_unfold(to_dev(x, dev), M, K, G, planes, amax)
    p_ref, a_ref = oracle.unfold(x, G, oracle.MODE_F)
    np.testing.assert_array_equal(amax.cpu().numpy(), a_ref.astype(np.float32))
    np.testing.assert_array_equal(planes.cpu().numpy(), p_ref)


# ------------------------------------------------------------------------------------------- step 9

PARTIAL_CASES = [
    # M, K, N, G, groups to check, x dist, w dist
    (1, 256, 128, 128, [0, 1], "normal", "u8"),
    (2, 512, 264, 32, [3, 15], "t3_clip60", "u8"),
    (2, 8320, 136, 64, [0, 129], "normal", "pm1_mix"),     # K > 8192: unfold kernel + streaming kernel
    (3, 512, 264, 64, [0, 5, 7], "t3_clip60", "u8"),
    (5, 96, 1000, 32, [0, 2], "normal", "u8"),
    (8, 1024, 384, 128, [3], "normal_cols20", "pm1_mix"),
    (16, 640, 136, 64, [9], "uniform3", "u7"),
    (17, 384, 256, 128, [2], "normal", "u8"),
    (40, 256, 128, 32, [0, 7], "normal", "u8"),
    # M >= 64: the unfold pre-pass and the 128 x 128 tile kernel
    (64, 512, 264, 64, [0, 5, 7], "t3_clip60", "u8"),
    (130, 384, 256, 128, [0, 2], "normal", "u8"),
    (200, 96, 1000, 32, [0, 2], "uniform3", "u7"),
    (256, 320, 136, 64, [4], "normal_cols20", "pm1_mix"),
]


@pytest.mark.parametrize("M,K,N,G,groups,xd,wd", PARTIAL_CASES)
def test_group_partials_bit_exact(dev, M, K, N, G, groups, xd, wd):
    x, wp, _ = I.make_inputs(I.small_case(M, K, N, G, seed=M * 7 + K, x_dist=xd, w_dist=wd))
    w_pre = wq.prepack_weight(to_dev(wp, dev), K, N, G)
    xdv = to_dev(x, dev)
    ws = wq.allocate_workspace(M, K, N, G, dev)
    for g in groups:
        y123 = torch.full((3, M, N), -12345, dtype=torch.int32, device=dev)
        wq.wqbmm_debug_group_partials(xdv, w_pre, M, K, N, G, g, y123, ws)
        np.testing.assert_array_equal(y123.cpu().numpy(), oracle.group_partials(x, wp, N, G, g, oracle.MODE_F),
                                      err_msg=f"group {g}")


@pytest.mark.parametrize("M", [4, 128])
@pytest.mark.parametrize("wval", [7, -8, 1, -1])
def test_group_partials_exact_at_extreme_magnitudes(dev, wval, M):
    """x constant per group gives planes (7, 7, 5) everywhere; with constant weights the integer sums reach the
    largest magnitudes the format allows (|Y| up to 7 * 8 * G), where inexact FP32 accumulation would show."""
    K, N, G = 256, 128, 128
    x = np.ones((M, K), dtype=np.float16)
    x[1] = -2.0
    x[2, :128] = 0.25
    w = np.full((K, N), wval, dtype=np.int8)
    wp = I.pack_int4_along_k(w)
    w_pre = wq.prepack_weight(to_dev(wp, dev), K, N, G)
    ws = wq.allocate_workspace(M, K, N, G, dev)
    for g in range(2):
        y123 = torch.zeros((3, M, N), dtype=torch.int32, device=dev)
        wq.wqbmm_debug_group_partials(to_dev(x, dev), w_pre, M, K, N, G, g, y123, ws)
        ref = oracle.group_partials(x, wp, N, G, g, oracle.MODE_F)
        np.testing.assert_array_equal(y123.cpu().numpy(), ref)


# ------------------------------------------------------------------------------------------- steps 1-11

RUN_CASES = [
    # M, K, N, G, x dist, w dist, scale lo, hi
    (1, 128, 128, 128, "normal", "u8", 0.005, 0.02),
    (3, 512, 264, 64, "t3_clip60", "u8", -1.0, 1.0),
    (5, 384, 136, 32, "normal", "u8", 0.005, 0.02),
    (7, 96, 1000, 32, "uniform3", "u7", -3.0, 3.0),
    (2, 8192, 128, 64, "normal", "u8", 0.001, 0.01),
    (12, 2048, 640, 128, "normal_cols20", "pm1_mix", 0.005, 0.02),
    (17, 640, 392, 64, "normal", "u8", 0.005, 0.02),
    (40, 1280, 520, 128, "t3_clip60", "u8", 0.002, 0.03),
    (64, 256, 128, 128, "normal", "u8", 0.005, 0.02),      # M >= 64: unfold pre-pass + 128 x 128 tiles
    (130, 512, 256, 64, "normal", "u8", 0.005, 0.02),
    (200, 96, 1000, 32, "uniform3", "u7", -3.0, 3.0),
    (256, 320, 392, 64, "t3_clip60", "u8", -1.0, 1.0),
    (300, 1280, 520, 128, "normal_cols20", "pm1_mix", 0.002, 0.03),
    (1, 65536, 256, 128, "normal", "u8", 0.005, 0.02),     # M <= 2, K > 8192: unfold kernel + streaming kernel
    (2, 8320, 264, 64, "t3_clip60", "u8", -1.0, 1.0),
    (2, 1024, 1000, 32, "uniform3", "u7", -3.0, 3.0),      # M <= 2, K <= 8192: one persistent kernel
    (2, 352, 136, 32, "normal", "u8", 0.005, 0.02),        # M <= 2, ragged last k-block (K = 2.75 x 128)
    (1, 1280, 39936, 128, "normal", "u8", 0.005, 0.02),    # M <= 2, 2496 column CTAs
    (3, 65536, 256, 128, "normal", "u8", 0.005, 0.02),     # 160-way split-K through the workspace
    (4, 4096, 1024, 128, "t3_clip60", "u8", -0.5, 0.5),    # 8 column tiles x 8 cluster slices
]


@pytest.mark.parametrize("M,K,N,G,xd,wd,lo,hi", RUN_CASES)
def test_run_matches_oracle(dev, M, K, N, G, xd, wd, lo, hi):
    x, wp, sc = I.make_inputs(I.small_case(M, K, N, G, seed=M + K + N, x_dist=xd, w_dist=wd, scale_lo=lo,
                                           scale_hi=hi))
    y = gpu_run(x, wp, sc, G, dev)
    T.assert_matches(y, oracle.msd_matmul(x, wp, sc, G, mode=oracle.MODE_D),
                     oracle.msd_matmul(x, wp, sc, G, mode=oracle.MODE_F), "run")


def test_run_zero_and_constant_rows(dev):
    M, K, N, G = 6, 512, 256, 128
    x, wp, sc = I.make_inputs(I.small_case(M, K, N, G, seed=3))
    x[0] = 0
    x[1, 128:256] = 0
    x[2] = np.float16(0.75)
    x[3, :128] = np.float16(-60.0)
    y = gpu_run(x, wp, sc, G, dev)
    assert not y[0].any()
    T.assert_matches(y, oracle.msd_matmul(x, wp, sc, G), oracle.msd_matmul(x, wp, sc, G, mode=oracle.MODE_F),
                     "special rows")


@pytest.mark.parametrize("wl", [I.WORKLOADS["decode_m1_k4096_n4096"],                  # cluster-reduced split-K
                                I.small_case(3, 16384, 520, 64, seed=8),               # workspace split-K
                                I.small_case(200, 1024, 392, 128, seed=9)])            # unfold pre-pass
def test_run_deterministic_and_workspace_left_clean(dev, wl):
    x, wp, sc = I.make_inputs(wl)
    xd, sd = to_dev(x, dev), to_dev(sc, dev)
    w_pre = wq.prepack_weight(to_dev(wp, dev), wl.K, wl.N, wl.G)
    ws = wq.allocate_workspace(wl.M, wl.K, wl.N, wl.G, dev)
    outs = []
    for _ in range(3):
        y = torch.empty((wl.M, wl.N), dtype=torch.float16, device=dev)
        wq.wqbmm_run(xd, w_pre, sd, y, wl.M, wl.K, wl.N, wl.G, ws)
        outs.append(y.cpu().numpy().view(np.uint16))
    assert all(np.array_equal(outs[0], o) for o in outs[1:])
    T.assert_matches(outs[0].view(np.float16), oracle.msd_matmul(x, wp, sc, wl.G),
                     oracle.msd_matmul(x, wp, sc, wl.G, mode=oracle.MODE_F), wl.name)
    if ws is not None and 2 < wl.M < 64:
        # the arrival counters sit after the partial sums; all must be back at zero
        counters = ws.cpu().numpy()[-256:].view(np.uint32)
        assert not counters.any()


@pytest.mark.parametrize("M,K,N,G", [(1, 4096, 520, 128), (2, 2048, 1000, 64), (1, 1024, 5120, 128)])
def test_calls_in_a_row_on_one_workspace(dev, M, K, N, G):
    """Calls in a row on one workspace with different x and no synchronisation between them: each result is its own
    x's, so a call's unfold pass never overwrites planes the previous call's GEMV kernel still reads, and a GEMV
    kernel never reads planes an earlier call left in the workspace (decode with a ragged N tile, two rows with
    G = 64, and an N with more CTAs than fit on the GPU at once)."""
    wl = I.small_case(M, K, N, G, seed=M + K + N)
    xa, wp, sc = I.make_inputs(wl)
    xb = I.make_x(I.small_case(M, K, N, G, seed=M + K + N + 1, x_dist="t3_clip60"))
    w_pre = wq.prepack_weight(to_dev(wp, dev), K, N, G)
    sd = to_dev(sc, dev)
    ws = wq.allocate_workspace(M, K, N, G, dev)
    xs = [xa, xb, xa, xb]
    ys = [torch.empty((M, N), dtype=torch.float16, device=dev) for _ in xs]
    xds = [to_dev(x, dev) for x in xs]
    for xd, y in zip(xds, ys):
        wq.wqbmm_run(xd, w_pre, sd, y, M, K, N, G, ws)
    torch.cuda.synchronize()
    for i, (x, y) in enumerate(zip(xs, ys)):
        T.assert_matches(y.cpu().numpy(), oracle.msd_matmul(x, wp, sc, G),
                         oracle.msd_matmul(x, wp, sc, G, mode=oracle.MODE_F), f"call {i}")


@pytest.mark.parametrize("wl", [I.small_case(1, 4096, 520, 128, seed=31),                   # decode
                                I.small_case(3, 16384, 520, 64, seed=32),                   # split-K, workspace
                                I.small_case(4, 4096, 1024, 128, seed=33),                  # split-K, cluster
                                I.small_case(130, 512, 256, 64, seed=34)])                  # large M
def test_run_needs_no_cleared_workspace(dev, wl):
    """A workspace full of leftover bytes (as an earlier run that gave up a wait could leave it) gives the same
    result: every kernel writes what it later reads, the split-K arrival counters included."""
    x, wp, sc = I.make_inputs(wl)
    w_pre = wq.prepack_weight(to_dev(wp, dev), wl.K, wl.N, wl.G)
    nbytes = wq.wqbmm_workspace_bytes(wl.M, wl.K, wl.N, wl.G)
    ws = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device=dev)
    y = torch.empty((wl.M, wl.N), dtype=torch.float16, device=dev)
    wq.wqbmm_run(to_dev(x, dev), w_pre, to_dev(sc, dev), y, wl.M, wl.K, wl.N, wl.G, ws)
    T.assert_matches(y.cpu().numpy(), oracle.msd_matmul(x, wp, sc, wl.G),
                     oracle.msd_matmul(x, wp, sc, wl.G, mode=oracle.MODE_F), "leftover workspace")


@pytest.mark.parametrize("M,K,N,G", [(1, 4096, 520, 128), (2, 1024, 264, 32), (5, 2048, 1000, 64),
                                     (3, 16384, 136, 128), (130, 512, 392, 64), (8, 1024, 264, 1024),
                                     (200, 256, 136, 256)])
def test_run_parts_compose_to_run(dev, M, K, N, G):
    """wqbmm_run_part: the pre-passes (part 1) and then the main kernel alone (part 2) give wqbmm_run's y bit for
    bit, on every path (per channel included); the main kernel alone again on the same workspace gives it too."""
    x, wp, sc = I.make_inputs(I.small_case(M, K, N, G, seed=M + 2 * K + N))
    xd, sd = to_dev(x, dev), to_dev(sc, dev)
    w_pre = wq.prepack_weight(to_dev(wp, dev), K, N, G)
    a = torch.empty((M, N), dtype=torch.float16, device=dev)
    wq.wqbmm_run(xd, w_pre, sd, a, M, K, N, G, wq.allocate_workspace(M, K, N, G, dev))
    ws = wq.allocate_workspace(M, K, N, G, dev)
    for parts in ((1, 2), (2,)):
        b = torch.full((M, N), 9.0, dtype=torch.float16, device=dev)
        for part in parts:
            wq.wqbmm_run_part(xd, w_pre, sd, None, None, b, M, K, N, G, ws, None, part)
        np.testing.assert_array_equal(a.cpu().numpy().view(np.uint16), b.cpu().numpy().view(np.uint16))


def test_run_errors_leave_output_untouched(dev):
    M, K, N, G = 1, 65536, 256, 128
    x, wp, sc = I.make_inputs(I.small_case(M, K, N, G, seed=5))
    xd, sd = to_dev(x, dev), to_dev(sc, dev)
    w_pre = wq.prepack_weight(to_dev(wp, dev), K, N, G)
    ws = wq.allocate_workspace(M, K, N, G, dev)
    y = torch.full((M, N), 7.0, dtype=torch.float16, device=dev)
    with pytest.raises(wq.WqbmmError) as e:
        wq.wqbmm_run(xd, w_pre, sd, y, M, K, N, G, ws, 64)                   # workspace too small
    assert e.value.status == wq.ERR_INVALID
    with pytest.raises(wq.WqbmmError) as e:
        wq.wqbmm_run(xd, w_pre, sd, y, M, K + 64, N, G, ws)                  # K not a multiple of G
    assert e.value.status == wq.ERR_INVALID
    torch.cuda.synchronize()
    assert (y == 7.0).all()


def test_bounded_wait_reports_timeout(dev):
    """A kernel waits on a barrier nothing completes; it gives up after 50 ms and records the timeout."""
    wq.wqbmm_debug_wait_timeout(50_000_000)
    code = wq.wqbmm_read_device_status(clear=True)
    assert code & 0xFF == wq.ERR_DEVICE_TIMEOUT and (code >> 8) == 9
    assert wq.wqbmm_read_device_status() == 0
    # the context is still usable
    x, wp, sc = I.make_inputs(I.small_case(2, 256, 128, 128, seed=1))
    T.assert_within_tolerance(gpu_run(x, wp, sc, 128, dev), oracle.msd_matmul(x, wp, sc, 128), "after timeout")


# ------------------------------------------------------------------------------------------- full workloads

@pytest.mark.parametrize("name", ["pr1_m16_k1024_n1024", "decode_m1_k4096_n4096", "ffn_up_m8_k4096_n11008",
                                  "page_sample_m1_k8192_n12288"])
def test_workload_full_output(dev, name):
    wl = I.WORKLOADS[name]
    x, wp, sc = I.make_inputs(wl)
    y = gpu_run(x, wp, sc, wl.G, dev)
    T.assert_matches(y, oracle.msd_matmul(x, wp, sc, wl.G, mode=oracle.MODE_D),
                     oracle.msd_matmul(x, wp, sc, wl.G, mode=oracle.MODE_F), name)


@pytest.mark.parametrize("name,nrows", [("mid_m128_k5120_n13824", 16), ("prefill_m2048_k8192_n28672", 64)])
def test_workload_sampled_rows(dev, name, nrows):
    wl = I.WORKLOADS[name]
    x, wp, sc = I.make_inputs(wl)
    y = gpu_run(x, wp, sc, wl.G, dev)
    rows = I.sample_rows(wl, nrows)
    T.assert_matches(y[rows], oracle.msd_matmul(x, wp, sc, wl.G, mode=oracle.MODE_D, rows=rows),
                     oracle.msd_matmul(x, wp, sc, wl.G, mode=oracle.MODE_F, rows=rows), name)
    # one group's integer partials on the same rows, bit-exact (the tensor-core step at full size)
    g = wl.groups // 2
    y123 = torch.empty((3, wl.M, wl.N), dtype=torch.int32, device=dev)
    w_pre = wq.prepack_weight(to_dev(wp, dev), wl.K, wl.N, wl.G)
    ws = wq.allocate_workspace(wl.M, wl.K, wl.N, wl.G, dev)
    wq.wqbmm_debug_group_partials(to_dev(x, dev), w_pre, wl.M, wl.K, wl.N, wl.G, g, y123, ws)
    got = y123.cpu().numpy()[:, rows]
    np.testing.assert_array_equal(got, oracle.group_partials(x, wp, wl.N, wl.G, g, oracle.MODE_F, rows=rows))


# ------------------------------------------------------------------------------------------- zero points, bias

EX_CASES = [
    # M, K, N, G, zero-point kind (None: no zero point), bias; covering every kernel path
    (1, 4096, 520, 128, "int", True),          # decode kernel, one row
    (2, 1024, 1000, 32, "frac", True),         # decode kernel, two rows, ragged last CTA
    (1, 65536, 256, 128, "frac", False),       # decode kernel, many passes
    (3, 512, 264, 64, "int", True),            # small-M tensor-core kernel
    (5, 384, 136, 32, "frac", True),
    (12, 2048, 640, 128, "int", False),
    (4, 4096, 1024, 128, "frac", True),        # cluster-reduced split-K
    (3, 65536, 256, 128, "frac", True),        # split-K through the workspace
    (17, 640, 392, 64, None, True),            # bias alone
    (40, 1280, 520, 128, "frac", False),
    (64, 256, 128, 128, "int", True),          # large-M: unfold pre-pass + 128 x 128 tiles
    (200, 96, 1000, 32, "frac", True),
    (256, 320, 392, 64, None, True),
    (300, 1280, 520, 128, "frac", False),
]


def gpu_run_ex(x, wp, sc, zp, bias, G, dev):
    M, K = x.shape
    N = sc.shape[1]
    w_pre = wq.prepack_weight(to_dev(wp, dev), K, N, G)
    y = wq.msd_matmul(to_dev(x, dev), w_pre, to_dev(sc, dev), G,
                      zero_point=None if zp is None else to_dev(zp, dev),
                      bias=None if bias is None else to_dev(bias, dev))
    return y.cpu().numpy()


@pytest.mark.parametrize("M,K,N,G,zkind,with_bias", EX_CASES)
def test_run_ex_matches_oracle(dev, M, K, N, G, zkind, with_bias):
    wl = I.small_case(M, K, N, G, seed=3 * M + K + N, x_dist="t3_clip60" if M % 2 else "normal")
    x, wp, sc = I.make_inputs(wl)
    zp = None if zkind is None else I.make_zero_point(wl, zkind)
    bias = I.make_bias(wl) if with_bias else None
    y = gpu_run_ex(x, wp, sc, zp, bias, G, dev)
    T.assert_matches(y, oracle.msd_matmul_ex(x, wp, sc, G, zero_point=zp, bias=bias, mode=oracle.MODE_D),
                     oracle.msd_matmul_ex(x, wp, sc, G, zero_point=zp, bias=bias, mode=oracle.MODE_F), "run_ex")


@pytest.mark.parametrize("M,K,N,G", [(1, 1024, 264, 64), (9, 1024, 264, 64), (130, 512, 256, 64)])
def test_run_ex_without_optionals_is_run(dev, M, K, N, G):
    """Null zero point and bias take the plain kernels: the output is the one of wqbmm_run, bit for bit."""
    x, wp, sc = I.make_inputs(I.small_case(M, K, N, G, seed=M + 40))
    xd, sd = to_dev(x, dev), to_dev(sc, dev)
    w_pre = wq.prepack_weight(to_dev(wp, dev), K, N, G)
    ws = wq.allocate_workspace(M, K, N, G, dev)
    a = torch.empty((M, N), dtype=torch.float16, device=dev)
    b = torch.empty((M, N), dtype=torch.float16, device=dev)
    wq.wqbmm_run(xd, w_pre, sd, a, M, K, N, G, ws)
    wq.wqbmm_run_ex(xd, w_pre, sd, None, None, b, M, K, N, G, ws)
    np.testing.assert_array_equal(a.cpu().numpy().view(np.uint16), b.cpu().numpy().view(np.uint16))


def test_run_ex_zero_zero_point_and_bias_change_nothing(dev):
    """zp = 0 and bias = 0 give the plain product (1 + 0/8 = 1 exactly; adding +0 keeps every nonzero value)."""
    M, K, N, G = 6, 1024, 392, 128
    x, wp, sc = I.make_inputs(I.small_case(M, K, N, G, seed=77))
    xd, sd = to_dev(x, dev), to_dev(sc, dev)
    w_pre = wq.prepack_weight(to_dev(wp, dev), K, N, G)
    ws = wq.allocate_workspace(M, K, N, G, dev)
    a = torch.empty((M, N), dtype=torch.float16, device=dev)
    b = torch.empty((M, N), dtype=torch.float16, device=dev)
    zeros_zp = torch.zeros((K // G, N), dtype=torch.float16, device=dev)
    zeros_b = torch.zeros(N, dtype=torch.float16, device=dev)
    wq.wqbmm_run(xd, w_pre, sd, a, M, K, N, G, ws)
    wq.wqbmm_run_ex(xd, w_pre, sd, zeros_zp, zeros_b, b, M, K, N, G, ws)
    np.testing.assert_array_equal(a.cpu().numpy().astype(np.float64), b.cpu().numpy().astype(np.float64))


def test_run_ex_rejects_unaligned_optionals(dev):
    M, K, N, G = 2, 256, 128, 128
    x, wp, sc = I.make_inputs(I.small_case(M, K, N, G, seed=4))
    xd, sd = to_dev(x, dev), to_dev(sc, dev)
    w_pre = wq.prepack_weight(to_dev(wp, dev), K, N, G)
    ws = wq.allocate_workspace(M, K, N, G, dev)
    y = torch.full((M, N), 7.0, dtype=torch.float16, device=dev)
    buf = torch.zeros(2 * N + 8, dtype=torch.float16, device=dev)
    for zp, bias in ((buf.data_ptr() + 2, None), (None, buf.data_ptr() + 2)):
        with pytest.raises(wq.WqbmmError) as e:
            wq.wqbmm_run_ex(xd, w_pre, sd, zp, bias, y, M, K, N, G, ws)
        assert e.value.status == wq.ERR_INVALID
    torch.cuda.synchronize()
    assert (y == 7.0).all()


def test_run_ex_mid_workload_sampled_rows(dev):
    """The mid-batch workload (M=128, K=5120, N=13824, G=128) with fractional zero points and a bias, through the
    large-M kernels, on sampled rows."""
    wl = I.WORKLOADS["mid_m128_k5120_n13824"]
    x, wp, sc = I.make_inputs(wl)
    zp, bias = I.make_zero_point(wl, "frac"), I.make_bias(wl)
    y = gpu_run_ex(x, wp, sc, zp, bias, wl.G, dev)
    rows = I.sample_rows(wl, 8)
    T.assert_matches(y[rows], oracle.msd_matmul_ex(x, wp, sc, wl.G, zero_point=zp, bias=bias, mode=oracle.MODE_D,
                                                   rows=rows),
                     oracle.msd_matmul_ex(x, wp, sc, wl.G, zero_point=zp, bias=bias, mode=oracle.MODE_F, rows=rows),
                     wl.name)


# ------------------------------------------------------------------------------------------- per channel (G = K)

PC_CASES = [
    # M, K, N, zero-point kind (None: none), bias
    (1, 4096, 520, None, False),      # decode kernel: one scale row serves every 128-k sub-group
    (2, 1024, 1000, "frac", True),
    (3, 2048, 264, None, False),      # small-M tensor-core kernel
    (8, 4096, 1000, "int", True),
    (16, 1024, 256, "frac", False),   # cluster-reduced split-K
    (3, 65536, 256, None, True),      # split-K through the workspace
    (64, 1024, 264, None, False),     # large-M pre-pass + tiles
    (130, 512, 256, "frac", True),
    (4, 352, 136, None, False),       # K not a multiple of 128: sub-groups of 32
    (200, 160, 264, "int", True),
]


@pytest.mark.parametrize("M,K,N,zkind,with_bias", PC_CASES)
def test_per_channel_matches_oracle(dev, M, K, N, zkind, with_bias):
    """G = K: A_max over each whole row, one scale (and zero-point) row; against the oracle run with one group."""
    wl = I.small_case(M, K, N, K, seed=5 * M + K + N, x_dist="t3_clip60" if M % 2 else "normal")
    x, wp, sc = I.make_inputs(wl)
    assert sc.shape == (1, N)
    zp = None if zkind is None else I.make_zero_point(wl, zkind)
    bias = I.make_bias(wl) if with_bias else None
    y = gpu_run_ex(x, wp, sc, zp, bias, K, dev)
    T.assert_matches(y, oracle.msd_matmul_ex(x, wp, sc, K, zero_point=zp, bias=bias, mode=oracle.MODE_D),
                     oracle.msd_matmul_ex(x, wp, sc, K, zero_point=zp, bias=bias, mode=oracle.MODE_F), "per channel")


@pytest.mark.parametrize("M,K", [(9, 1024), (3, 352), (2, 4096)])
def test_unfold_bit_exact_per_channel(dev, M, K):
    x = I.make_x(I.small_case(M, K, 8, K, seed=K + M, x_dist="t3_clip60"))
    planes = torch.empty((3, M, K), dtype=torch.int8, device=dev)
    amax = torch.empty((M, 1), dtype=torch.float32, device=dev)
    wq.wqbmm_debug_unfold(to_dev(x, dev), M, K, K, planes, amax)
    p_ref, a_ref = oracle.unfold(x, K, oracle.MODE_F)
    np.testing.assert_array_equal(amax.cpu().numpy(), a_ref.astype(np.float32))
    np.testing.assert_array_equal(planes.cpu().numpy(), p_ref)


# ------------------------------------------------------------------------------------------- batched x, shared weights

@pytest.mark.parametrize("B,M,K,N,G", [(3, 5, 1024, 264, 64), (2, 1, 4096, 520, 128), (4, 40, 512, 256, 128)])
def test_batched_x_matches_oracle(dev, B, M, K, N, G):
    """x [B, M, K] with one weight: the binding folds the batch into rows; the oracle sees the same rows."""
    wl = I.small_case(B * M, K, N, G, seed=B * 100 + M)
    x, wp, sc = I.make_inputs(wl)
    w_pre = wq.prepack_weight(to_dev(wp, dev), K, N, G)
    y = wq.msd_matmul(to_dev(x.reshape(B, M, K), dev), w_pre, to_dev(sc, dev), G)
    assert tuple(y.shape) == (B, M, N)
    T.assert_matches(y.cpu().numpy(), oracle.msd_matmul(x, wp, sc, G, mode=oracle.MODE_D).reshape(B, M, N),
                     oracle.msd_matmul(x, wp, sc, G, mode=oracle.MODE_F).reshape(B, M, N), "batched")


@pytest.mark.parametrize("B,M,K,N,G", [(3, 5, 1024, 264, 64), (2, 70, 256, 128, 128)])
def test_batched_strided_matches_oracle(dev, B, M, K, N, G):
    """Batches with gaps between them (x padded by 2 rows, y by 1 row per item): each item is its own product, the
    gaps of y stay untouched; the contiguous form of the same batch equals one product of B * M rows bit for bit."""
    wl = I.small_case(B * M, K, N, G, seed=B * 7 + M)
    x, wp, sc = I.make_inputs(wl)
    zp, bias = I.make_zero_point(wl, "frac"), I.make_bias(wl)
    w_pre = wq.prepack_weight(to_dev(wp, dev), K, N, G)
    xpad = np.zeros((B, M + 2, K), dtype=np.float16)
    xpad[:, :M] = x.reshape(B, M, K)
    xd = to_dev(xpad, dev)
    y = torch.full((B, M + 1, N), 3.0, dtype=torch.float16, device=dev)
    ws = wq.allocate_workspace(M, K, N, G, dev)
    wq.wqbmm_run_batched(xd, w_pre, to_dev(sc, dev), to_dev(zp, dev), to_dev(bias, dev), y, B, M, K, N, G,
                         (M + 2) * K, (M + 1) * N, ws)
    got = y.cpu().numpy()
    assert (got[:, M] == 3.0).all()
    for b in range(B):
        xb = x[b * M:(b + 1) * M]
        T.assert_matches(got[b, :M], oracle.msd_matmul_ex(xb, wp, sc, G, zero_point=zp, bias=bias, mode=oracle.MODE_D),
                         oracle.msd_matmul_ex(xb, wp, sc, G, zero_point=zp, bias=bias, mode=oracle.MODE_F),
                         f"item {b}")
    # contiguous: one product of B * M rows
    xc = to_dev(x, dev)
    yc = torch.empty((B * M, N), dtype=torch.float16, device=dev)
    yo = torch.empty((B * M, N), dtype=torch.float16, device=dev)
    wsc = wq.allocate_workspace(B * M, K, N, G, dev)
    wq.wqbmm_run_batched(xc, w_pre, to_dev(sc, dev), None, None, yc, B, M, K, N, G, M * K, M * N, wsc)
    wq.wqbmm_run(xc, w_pre, to_dev(sc, dev), yo, B * M, K, N, G, wsc)
    np.testing.assert_array_equal(yc.cpu().numpy().view(np.uint16), yo.cpu().numpy().view(np.uint16))


# ------------------------------------------------------------------------------------------- int8 weights (W8)

def split_w8_packed(w8, G):
    """The int4 form of int8 weights as documented for wqbmm_run_w8, restated with numpy: group g of w becomes
    groups 2g (hi = w >> 4) and 2g + 1 (lo - 8 with lo = w & 15) of a [2K, N] int4 matrix, packed along k."""
    K, N = w8.shape
    w16 = w8.astype(np.int16)
    hi = (w16 >> 4).reshape(K // G, G, N)
    lo = ((w16 & 15) - 8).reshape(K // G, G, N)
    return I.pack_int4_along_k(np.stack([hi, lo], axis=1).reshape(2 * K, N).astype(np.int8))


@pytest.mark.parametrize("K,N,G", [(256, 128, 128), (640, 264, 64), (96, 1000, 32)])
def test_prepack_w8_is_the_documented_split(dev, K, N, G):
    w8 = I.make_w8(I.small_case(1, K, N, G, seed=K + N))
    a = wq.prepack_weight_w8(to_dev(w8, dev), K, N, G).cpu().numpy()
    b = wq.prepack_weight(to_dev(split_w8_packed(w8, G), dev), 2 * K, N, G).cpu().numpy()
    np.testing.assert_array_equal(a, b)


W8_CASES = [
    # M, K, N, G, zero-point kind, bias
    (1, 4096, 520, 128, None, False),       # decode kernel
    (2, 1024, 1000, 32, "frac", True),
    (3, 2048, 264, 64, None, True),         # small-M tensor-core kernel
    (8, 4096, 1000, 128, "int", False),
    (16, 1024, 256, 128, "frac", True),
    (64, 512, 264, 64, None, False),        # large-M
    (130, 384, 256, 128, "int", True),
]


@pytest.mark.parametrize("M,K,N,G,zkind,with_bias", W8_CASES)
def test_w8_matches_oracle(dev, M, K, N, G, zkind, with_bias):
    wl = I.small_case(M, K, N, G, seed=11 * M + K + N, x_dist="t3_clip60" if M % 2 else "normal")
    x = I.make_x(wl)
    sc = I.make_scale(wl)
    w8 = I.make_w8(wl)
    zp = None if zkind is None else (I.make_zero_point(wl, zkind) * 16).astype(np.float16)   # int8 range
    bias = I.make_bias(wl) if with_bias else None
    w_pre = wq.prepack_weight_w8(to_dev(w8, dev), K, N, G)
    y = wq.msd_matmul_w8(to_dev(x, dev), w_pre, to_dev(sc, dev), G,
                         zero_point=None if zp is None else to_dev(zp, dev),
                         bias=None if bias is None else to_dev(bias, dev)).cpu().numpy()
    T.assert_matches(y, oracle.msd_matmul_w8(x, w8, sc, G, zero_point=zp, bias=bias, mode=oracle.MODE_D),
                     oracle.msd_matmul_w8(x, w8, sc, G, zero_point=zp, bias=bias, mode=oracle.MODE_F), "int8 weights")
