"""Benchmark of the A16W4 per-group MSD matmul on GB300.

One step = one wqbmm_run over one batch of the workload: all steps of the method (A_max, unfold, the three integer
matmuls, the per-group combine, the accumulation and the fp16 store). Every path is an unfold pre-pass followed by
the main kernel (M <= 2: dp4a matrix-vector kernel; 3 <= M < 64: small-M tensor-core kernel; M >= 64: tensor-core
tile kernel).

Default workload: decode GEMV M=1, K=4096, N=4096, G=128 (x ~ N(0,1) fp16, int4 weights uniform on [-8, 7],
antiquant_scale uniform on [0.005, 0.02], seed 1). Metric: effective weight GB/s (K*N/2 bytes per step / step time)
for M <= 16, int8-equivalent TOPS (6 M N K per step / step time) above.

Timing: W warm-up steps, then a short sustained phase (not timed, keeps the clocks representative and gives the
clock sampler something to see), then exactly K timed steps between CUDA events on the launching stream, replayed
from CUDA graphs (a short device-side spin before the start event keeps the host's graph-launch latency out of the
timed region); then K launches of the main kernel alone (wqbmm_run_part, part 2), the same way, for the roofline
of the dominant kernel. Each step uses a different copy of the weights, scales and input (rotating copies whose total
is more than twice the 126 MB L2), so every step streams its weights from HBM. The other workload shapes are timed
the same way into a `workloads` record of the same line. The dense tensor-core peaks (E4M3, int8, bf16) are measured
in the same run; the E4M3 one is the denominator of the tensor-bound fractions.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

With N > 1 (torchrun), each rank runs an independent replica on its own GPU (the operation has no exchange step);
ranks meet at a barrier around the timed region and the slowest rank's time is used. `--impl reference` times the
CPU oracle (the plain C implementation of the method used by the tests) on the host cores instead.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from weight_quantized_matmul_gb300 import inputs as I  # noqa: E402

DEFAULT_WORKLOAD = "decode_m1_k4096_n4096"
L2_BYTES = 126 * 1024 * 1024
HOLD_CYCLES = 200_000            # ~0.1 ms of device spin before each timed region
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(I.WORKLOADS))
    ap.add_argument("--impl", default="wqbmm", choices=["wqbmm", "reference"])
    ap.add_argument("--zero-point", default="none", choices=["none", "int", "frac"],
                    help="asymmetric weights: seeded zero points [K/G, N] (wqbmm_run_ex)")
    ap.add_argument("--bias", action="store_true", help="add a seeded bias [N] (wqbmm_run_ex)")
    ap.add_argument("--per-channel", action="store_true", help="per-channel quantization: G = K, scale [1, N]")
    ap.add_argument("--w8", action="store_true", help="int8 weights [K, N] (wqbmm_run_w8)")
    ap.add_argument("--sustain-s", type=float, default=1.5)
    ap.add_argument("--cpu-baseline-s", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="time only the selected workload")
    return ap.parse_args()


def metric_for(wl):
    if wl.M <= 16:
        return "A16W4 MSD matmul weight GB/s (M<=16)", "GB/s"
    return "A16W4 MSD matmul int8-equivalent TOPS (6*M*N*K)", "TOPS"


def units_per_step(wl, w8=False):
    """The metric's numerator for one step: weight bytes (M<=16; int8 weights take K N bytes) or int8-equivalent
    ops."""
    if wl.M <= 16:
        return wl.K * wl.N if w8 else wl.weight_bytes()
    return wl.int8_equiv_ops()


def metric_value(wl, seconds_per_step, n=1, w8=False):
    return n * units_per_step(wl, w8) / seconds_per_step / (1e9 if wl.M <= 16 else 1e12)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS}, "fallback"


def slowest_rank_ms(ms_total, world, device=None):
    """The timed region's length on the slowest rank (every rank calls this; NCCL reduces on the GPU, gloo on the
    host)."""
    if world <= 1:
        return ms_total
    import torch
    import torch.distributed as dist
    on = device if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([ms_total], dtype=torch.float64, device=on)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def kernel_sources_hash():
    """Hash of the CUDA sources the library is built from (names and contents, in name order)."""
    import hashlib
    h = hashlib.sha256()
    src = os.path.join(ROOT, "weight_quantized_matmul_gb300", "csrc")
    for name in sorted(os.listdir(src)):
        if name.endswith((".cu", ".cuh")):
            h.update(name.encode())
            with open(os.path.join(src, name), "rb") as f:
                h.update(f.read())
    return h.hexdigest()


def dram_traffic(workload):
    """DRAM bytes per launch of the workload's dominant kernel from the committed ncu capture, or None when there
    is none or the kernel sources changed since it was taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            table = json.load(f)
    except (OSError, ValueError):
        return None
    rec = table.get("workloads", {}).get(workload)
    if not rec or table.get("kernel_sources_sha256") != kernel_sources_hash():
        return None
    return rec.get("dram_bytes_per_launch")


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def nvsmi_id(torch, dev, local):
    """The identifier nvidia-smi needs for this process's GPU (its UUID when torch knows it)."""
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        if uuid:
            return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        pass
    visible = os.environ.get("CUDA_VISIBLE_DEVICES")
    if visible:
        return visible.split(",")[local].strip()
    return str(local)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.time(), ln.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0=None, t1=None):
        """Median SM clock, maximum and throttle reasons seen over the samples taken between t0 and t1 (all when
        not given)."""
        sm, smax, reasons = [], 0.0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for t, ln in self.lines:
            if (t0 is not None and t < t0) or (t1 is not None and t > t1):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = max(smax, float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def _oracle_blocks(wl, x, wp, sc, rows, threads):
    """The oracle's work split into `threads` independent calls: blocks of output columns (their weight columns and
    scales copied out once), all rows (or the seeded rows) each."""
    n_blocks = max(1, min(threads, wl.N // 8))
    edges = [wl.N * i // n_blocks // 8 * 8 for i in range(n_blocks)] + [wl.N]
    blocks = []
    for a, b in zip(edges[:-1], edges[1:]):
        if b > a:
            blocks.append((np.ascontiguousarray(wp[:, a:b]), np.ascontiguousarray(sc[:, a:b])))
    return blocks


def cpu_oracle_baseline(wl, budget_s, threads=1):
    """The oracle as it stands (binary64 MSD, plain C) on the workload: whole problems, or seeded rows when one
    problem would be too long for the budget. With threads > 1 the calls run on that many host threads at once,
    each on its own block of output columns (the oracle releases the interpreter lock while it computes). Returns
    the metric value, the threads used, a description of the sample and the seconds per problem sample."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    x, wp, sc = I.make_inputs(wl)
    rows = I.sample_rows(wl, 8) if wl.M > 16 else None
    nrows = len(rows) if rows is not None else wl.M
    per_row_units = units_per_step(wl) / wl.M
    blocks = _oracle_blocks(wl, x, wp, sc, rows, threads)

    def one_block(b):
        oracle.msd_matmul(x, b[0], b[1], wl.G, mode=oracle.MODE_D, rows=rows)

    pool = ThreadPoolExecutor(max_workers=len(blocks)) if len(blocks) > 1 else None
    t0 = time.perf_counter()
    calls = 0
    while True:
        if pool is None:
            one_block(blocks[0])
        else:
            list(pool.map(one_block, blocks))
        calls += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = (time.perf_counter() - t0) / calls
    if pool is not None:
        pool.shutdown()
    value = per_row_units * nrows / dt / (1e9 if wl.M <= 16 else 1e12)
    what = f"the whole {wl.name} problem" if rows is None else f"{nrows} seeded rows of {wl.name}"
    sample = f"{calls} passes over {what}, {len(blocks)} column block(s) on {len(blocks)} thread(s)"
    return value, len(blocks), sample, dt


def run_reference(args, wl):
    """The reference arm: the oracle, as it stands, on all host cores (column blocks on threads), timed per step."""
    world, rank, _ = dist_env()
    if world > 1 and rank != 0:
        return
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    metric, unit = metric_for(wl)
    x, wp, sc = I.make_inputs(wl)
    rows = I.sample_rows(wl, 8) if wl.M > 16 else None
    nrows = len(rows) if rows is not None else wl.M
    units = units_per_step(wl) / wl.M * nrows
    blocks = _oracle_blocks(wl, x, wp, sc, rows, os.cpu_count() or 1)
    pool = ThreadPoolExecutor(max_workers=len(blocks))

    def step():
        list(pool.map(lambda b: oracle.msd_matmul(x, b[0], b[1], wl.G, mode=oracle.MODE_D, rows=rows), blocks))

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    pool.shutdown()
    value = units / dt / (1e9 if wl.M <= 16 else 1e12)
    sample = ("whole problem per step" if rows is None else f"{nrows} seeded rows per step") + \
        f", {len(blocks)} column blocks on {len(blocks)} threads"
    print(json.dumps({
        "impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "M": wl.M, "K": wl.K, "N": wl.N, "G": wl.G,
                   "parallelism": f"host cores, {len(blocks)} threads"},
        "cpu_baseline": {"value": value, "unit": unit, "cores": len(blocks), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def tensor_peaks(torch, dev, n=8192, reps=10):
    """Dense tensor-core peaks measured here, best of `reps` n^3 products (CUDA events): E4M3 through
    torch._scaled_mm (the format this path's MMAs use), int8 through torch._int_mm, bf16 through torch.matmul."""
    out = {"shape": f"{n}^3, best of {reps}"}

    def best(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        t = float("inf")
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            t = min(t, a.elapsed_time(b))
        return 2.0 * n ** 3 / (t * 1e-3) / 1e12

    try:
        a8 = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        b8 = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()
        one = torch.tensor(1.0, device=dev)
        out["e4m3_tflops"] = best(lambda: torch._scaled_mm(a8, b8, scale_a=one, scale_b=one, out_dtype=torch.bfloat16))
        del a8, b8
    except Exception as e:                      # noqa: BLE001 - report, fall back to the bf16 ratio
        out["e4m3_error"] = repr(e)[:160]
    try:
        ai = torch.randint(-8, 8, (n, n), device=dev, dtype=torch.int8)
        bi = torch.randint(-8, 8, (n, n), device=dev, dtype=torch.int8)
        out["int8_tops"] = best(lambda: torch._int_mm(ai, bi))
        del ai, bi
    except Exception as e:                      # noqa: BLE001
        out["int8_error"] = repr(e)[:160]
    ah = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
    out["bf16_tflops"] = best(lambda: ah @ ah)
    del ah
    torch.cuda.empty_cache()
    return out


def measure(torch, wq, wl, args, dev, sampler, steps, sustain_s, variant, with_e2e):
    """Times `steps` calls of the workload replayed from CUDA graphs (the whole call, and the main kernel alone),
    with rotating input copies larger than twice L2, after warm-up and a sustained phase. Returns a record."""
    zero_point, bias, w8 = variant
    x, wp, sc = I.make_inputs(wl)
    if w8:
        wp = I.make_w8(wl)
    per_copy = wp.nbytes + x.nbytes + sc.nbytes
    copies = max(2, min(64, -(-2 * L2_BYTES // per_copy)))
    xd = torch.from_numpy(x).to(dev)
    sd = torch.from_numpy(sc).to(dev)
    wd = torch.from_numpy(wp).to(dev)
    w_pre0 = wq.prepack_weight_w8(wd, wl.K, wl.N, wl.G) if w8 else wq.prepack_weight(wd, wl.K, wl.N, wl.G)
    del wd
    w_pre = [w_pre0] + [w_pre0.clone() for _ in range(copies - 1)]
    xs = [xd] + [xd.clone() for _ in range(copies - 1)]
    ss = [sd] + [sd.clone() for _ in range(copies - 1)]
    ys = [torch.empty((wl.M, wl.N), dtype=torch.float16, device=dev) for _ in range(copies)]
    if w8:
        ws = [torch.zeros(wq.wqbmm_workspace_bytes_w8(wl.M, wl.K, wl.N, wl.G), dtype=torch.uint8, device=dev)
              for _ in range(copies)]
    else:
        ws = [wq.allocate_workspace(wl.M, wl.K, wl.N, wl.G, dev) for _ in range(copies)]
    zs = [None] * copies
    if zero_point != "none":
        zd = torch.from_numpy(I.make_zero_point(wl, zero_point)).to(dev)
        zs = [zd] + [zd.clone() for _ in range(copies - 1)]
    bd = torch.from_numpy(I.make_bias(wl)).to(dev) if bias else None
    stream = torch.cuda.Stream(device=dev)

    def step(i, s, part=0):
        c = i % copies
        if w8:
            wq.wqbmm_run_w8(xs[c], w_pre[c], ss[c], zs[c], bd, ys[c], wl.M, wl.K, wl.N, wl.G, ws[c], None, s)
        else:
            wq.wqbmm_run_part(xs[c], w_pre[c], ss[c], zs[c], bd, ys[c], wl.M, wl.K, wl.N, wl.G, ws[c], None, part,
                              s)

    # warm-up (eager; also sets kernel attributes before any capture), then one call per copy so that every
    # workspace holds its copy's unfolded x for the main-kernel-only graph
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i, stream)
        for c in range(copies):
            step(c, stream)
    torch.cuda.synchronize()
    if wq.wqbmm_read_device_status(stream=stream) != 0:
        raise SystemExit("device status error during warm-up")

    chunk = min(steps, 4 * copies)

    def graphs_for(part):
        made = {}

        def graph(n):
            if n not in made:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for i in range(n):
                        step(i, torch.cuda.current_stream(), part)
                made[n] = g
            return made[n]
        full, rem = divmod(steps, chunk)
        return graph(chunk), (graph(rem) if rem else None), full

    def timed(gfull, grem, full):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            # a short spin on the device holds the stream while the host queues the graph replays, so that the start
            # event is followed at once by the first step rather than by the host's launch latency
            torch.cuda._sleep(HOLD_CYCLES)
            a.record(stream)
            for _ in range(full):
                gfull.replay()
            if grem is not None:
                grem.replay()
            b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    g_call = graphs_for(0)
    g_main = None if w8 else graphs_for(2)
    torch.cuda.synchronize()
    t_start = time.time()
    t_end = t_start + sustain_s
    with torch.cuda.stream(stream):                 # sustained phase: steady clocks, clock samples around the timing
        while time.time() < t_end:
            g_call[0].replay()
            stream.synchronize()
    world = dist_env()[0]
    if world > 1:
        torch.distributed.barrier()
    ms_total = timed(*g_call)
    if world > 1:
        torch.distributed.barrier()
    main_ms = timed(*g_main) if g_main is not None else None
    t_stop = time.time()
    status = wq.wqbmm_read_device_status(stream=stream)
    if status != 0:
        raise SystemExit(f"device status error {status:#x}")
    rec = {"ms_total": ms_total, "ms_step": ms_total / steps, "steps": steps, "copies": copies,
           "per_copy": per_copy, "chunk": chunk,
           "kernel_us": None if main_ms is None else main_ms / steps * 1e3,
           "clocks": sampler.summary(t_start, t_stop), "x_bytes": int(x.nbytes)}
    if with_e2e:
        # end to end through the C ABI with host buffers: pinned x in, pinned y out, every step
        x_host = torch.from_numpy(x).pin_memory()
        y_host = torch.empty((wl.M, wl.N), dtype=torch.float16).pin_memory()
        e2e_steps = max(20, min(steps, 500))
        with torch.cuda.stream(stream):
            for i in range(3):
                xs[0].copy_(x_host, non_blocking=True)
                step(0, stream)
                y_host.copy_(ys[0], non_blocking=True)
                stream.synchronize()
            t0 = time.perf_counter()
            for i in range(e2e_steps):
                c = i % copies
                xs[c].copy_(x_host, non_blocking=True)
                step(c, stream)
                y_host.copy_(ys[c], non_blocking=True)
                stream.synchronize()
            rec["e2e_s"] = (time.perf_counter() - t0) / e2e_steps
    del w_pre, xs, ss, ys, ws, zs
    torch.cuda.empty_cache()
    return rec


def roofline_for(wl, rec, peaks, peak_kind, alg_bytes, variant_name):
    """Roofline of the dominant (main) kernel: algorithmic bytes (M <= 16) or int8-equivalent ops per call over the
    main kernel's own time per launch (timed alone, CUDA events over a graph of main-kernel launches); the same
    figure over the whole call (pre-passes included) as call_frac."""
    call_s = rec["ms_step"] * 1e-3
    kern_s = rec["kernel_us"] * 1e-6 if rec["kernel_us"] else None
    if wl.M <= 16:
        peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
        work, unit, bound, div = alg_bytes, "GB/s", "hbm", 1e9
        source = f"{peak_kind} hbm_gbs"
    else:
        e4m3 = peaks.get("e4m3_tflops")
        if e4m3:
            peak, source = e4m3, "e4m3 dense, torch._scaled_mm measured in this run"
        else:
            peak = 2 * float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
            source = f"{peak_kind} bf16_tflops x 2 (nominal e4m3 : bf16 ratio)"
        work, unit, bound, div = wl.int8_equiv_ops(), "TFLOP/s", "tensor", 1e12
    achieved = work / (kern_s if kern_s else call_s) / div
    call_achieved = work / call_s / div
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
            "traffic": None if variant_name else dram_traffic(wl.name),
            "kernel_us": rec["kernel_us"], "call_us": rec["ms_step"] * 1e3,
            "call_achieved": call_achieved, "call_frac": call_achieved / peak,
            "peak_source": source,
            ("algorithmic_bytes_per_launch" if bound == "hbm" else "algorithmic_flops_per_launch"): work}


def main():
    args = parse()
    wl = I.WORKLOADS[args.workload]
    if args.per_channel:
        wl = dataclasses.replace(wl, G=wl.K)
    if args.impl == "reference":
        run_reference(args, wl)
        return

    import torch

    import weight_quantized_matmul_gb300 as wq
    from weight_quantized_matmul_gb300 import build as wqbuild

    world, rank, local = dist_env()
    if args.warmup < 3:
        raise SystemExit("at least 3 warm-up steps")
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    wqbuild.build()
    metric, unit = metric_for(wl)

    sampler = ClockSampler(nvsmi_id(torch, dev, local))
    sampler.start()
    variant = (args.zero_point, bool(args.bias), bool(args.w8))
    variant_name = ",".join(n for n, on in (("zero_point", args.zero_point != "none"), ("bias", args.bias),
                                             ("per_channel", args.per_channel), ("w8", args.w8)) if on)
    rec = measure(torch, wq, wl, args, dev, sampler, args.steps, args.sustain_s, variant, True)
    ms_step = slowest_rank_ms(rec["ms_total"], world, dev) / args.steps

    others = {}
    if not variant_name and not args.no_workloads:
        # every other workload shape of the metric, shorter sustained phase, same steps (at least 10)
        for name, other in I.WORKLOADS.items():
            if name == wl.name:
                continue
            r = measure(torch, wq, other, args, dev, sampler, max(10, args.steps), 0.5, variant, False)
            others[name] = r
    peaks_here = tensor_peaks(torch, dev) if rank == 0 else {}
    time.sleep(0.25)
    sampler.stop()
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    peaks, peak_kind = measured_peaks()
    peaks = dict(peaks)
    if "e4m3_tflops" in peaks_here:
        peaks["e4m3_tflops"] = peaks_here["e4m3_tflops"]
    # the optional inputs add their own bytes: zero points 2 (K/G) N, bias 2 N
    alg_bytes = (wl.algorithmic_bytes() + (2 * wl.groups * wl.N if args.zero_point != "none" else 0) +
                 (2 * wl.N if args.bias else 0) + (wl.K * wl.N // 2 if args.w8 else 0))
    rec["ms_step"] = ms_step
    roofline = roofline_for(wl, rec, peaks, peak_kind, alg_bytes, variant_name)
    launches_per_step = 2 + (1 if args.per_channel or args.w8 else 0)
    line = {
        "metric": metric,
        "value": metric_value(wl, ms_step * 1e-3, world, args.w8),
        "unit": unit,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        # the arithmetic of the path this workload takes: dp4a on the CUDA cores for M <= 2, tensor cores above
        "dtype": ("fp16 x / int4 w -> int8 planes, dp4a int32 products, f32 epilogue" if wl.M <= 2 else
                  "fp16 x / int4 w -> e4m3 tensor-core MMA, f32 accumulate and epilogue"),
        "data": "synthetic",
        "config": {"workload": wl.name, "M": wl.M, "K": wl.K, "N": wl.N, "G": wl.G,
                   "zero_point": args.zero_point, "bias": bool(args.bias), "per_channel": bool(args.per_channel),
                   "weights": "int8" if args.w8 else "int4",
                   "parallelism": f"replicas{world}" if world > 1 else "single GPU",
                   "l2": f"{rec['copies']} rotating input copies ({rec['copies'] * rec['per_copy'] / 2**20:.0f} MiB "
                         f"> 2x L2)",
                   "launch": f"CUDA graphs of {rec['chunk']} steps"},
        "gpu_launches": args.steps * launches_per_step,
        "clocks": rec["clocks"],
        "e2e": {"value": metric_value(wl, rec["e2e_s"], 1, args.w8), "unit": unit,
                "h2d_bytes_per_step": rec["x_bytes"], "d2h_bytes_per_step": int(wl.M * wl.N * 2),
                "note": "eager wqbmm_run per step; pinned x in, pinned y out, stream synchronized each step"},
        "roofline": roofline,
        "tensor_peaks": peaks_here,
    }
    if others:
        recs = {}
        for name, r in others.items():
            owl = I.WORKLOADS[name]
            om, ou = metric_for(owl)
            rf = roofline_for(owl, r, peaks, peak_kind, owl.algorithmic_bytes(), "")
            recs[name] = {"metric": om, "value": metric_value(owl, r["ms_step"] * 1e-3), "unit": ou,
                          "ms": r["ms_step"], "kernel_us": r["kernel_us"], "steps": r["steps"],
                          "frac": rf["frac"], "call_frac": rf["call_frac"], "bound": rf["bound"],
                          "peak": rf["peak"], "traffic": rf["traffic"], "clocks": r["clocks"]}
        line["workloads"] = recs
    if not args.no_cpu_baseline:
        v1, c1, sample1, dt1 = cpu_oracle_baseline(wl, args.cpu_baseline_s / 2, threads=1)
        vn, cn, samplen, dtn = cpu_oracle_baseline(wl, args.cpu_baseline_s / 2, threads=os.cpu_count() or 1)
        line["cpu_baseline"] = {"value": vn, "unit": unit, "cores": cn, "kind": "oracle", "sample": samplen,
                                "s_per_call": dtn, "single_thread": {"value": v1, "cores": c1, "sample": sample1,
                                                                     "s_per_call": dt1}}
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
