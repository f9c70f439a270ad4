"""Benchmark of the A16W4 per-group MSD matmul on GB300.

One step = one wqbmm_run over one batch of the workload: all steps of the method (A_max, unfold, the three integer
matmuls, the per-group combine, the accumulation and the fp16 store). Depending on M that is one fused kernel
(3 <= M < 64) or an unfold kernel followed by the main kernel (M <= 2: dp4a matrix-vector kernel; M >= 64:
tensor-core tile kernel).

Default workload: decode GEMV M=1, K=4096, N=4096, G=128 (x ~ N(0,1) fp16, int4 weights uniform on [-8, 7],
antiquant_scale uniform on [0.005, 0.02], seed 1). Metric: effective weight GB/s (K*N/2 bytes per step / step time).

Timing: W warm-up steps, then a short sustained phase (not timed, keeps the clocks representative and gives the
clock sampler something to see), then exactly K timed steps between CUDA events on the launching stream, replayed
from CUDA graphs. Each step uses a different copy of the weights, scales and input (rotating copies whose total is
more than twice the 126 MB L2), so every step streams its weights from HBM.

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

    def summary(self):
        sm, smax, reasons = [], 0.0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for _, ln in self.lines:
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


def cpu_oracle_baseline(wl, budget_s):
    """The oracle as it stands (binary64 MSD, single thread) on whole problems of the workload, or on seeded rows
    when one problem alone would exceed the budget. Returns the metric value and a description."""
    import oracle
    x, wp, sc = I.make_inputs(wl)
    rows = None
    per_row_units = units_per_step(wl) / wl.M
    if wl.M > 16:
        rows = I.sample_rows(wl, 8)
    t0 = time.perf_counter()
    calls = 0
    while True:
        oracle.msd_matmul(x, wp, sc, wl.G, mode=oracle.MODE_D, rows=rows)
        calls += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = (time.perf_counter() - t0) / calls
    units = per_row_units * (len(rows) if rows is not None else wl.M)
    value = units / dt / (1e9 if wl.M <= 16 else 1e12)
    sample = (f"{calls} calls of the whole {wl.name} problem" if rows is None else
              f"{calls} calls on {len(rows)} seeded rows of {wl.name}")
    return value, 1, sample, dt


def run_reference(args, wl):
    world, rank, _ = dist_env()
    if world > 1 and rank != 0:
        return
    import oracle
    metric, unit = metric_for(wl)
    x, wp, sc = I.make_inputs(wl)
    rows = I.sample_rows(wl, 8) if wl.M > 16 else None
    nrows = len(rows) if rows is not None else wl.M
    units = units_per_step(wl) / wl.M * nrows
    for _ in range(args.warmup):
        oracle.msd_matmul(x, wp, sc, wl.G, mode=oracle.MODE_D, rows=rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.msd_matmul(x, wp, sc, wl.G, mode=oracle.MODE_D, rows=rows)
    dt = (time.perf_counter() - t0) / args.steps
    value = units / dt / (1e9 if wl.M <= 16 else 1e12)
    sample = "whole problem per step" if rows is None else f"{nrows} seeded rows per step"
    print(json.dumps({
        "impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "M": wl.M, "K": wl.K, "N": wl.N, "G": wl.G,
                   "parallelism": "host cores, single thread"},
        "cpu_baseline": {"value": value, "unit": unit, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


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

    # ---- inputs: host copy once, then rotating device copies whose total exceeds 2x L2
    x, wp, sc = I.make_inputs(wl)
    if args.w8:
        wp = I.make_w8(wl)
    per_copy = wp.nbytes + x.nbytes + sc.nbytes
    copies = max(2, min(64, -(-2 * L2_BYTES // per_copy)))
    xd = torch.from_numpy(x).to(dev)
    sd = torch.from_numpy(sc).to(dev)
    wd = torch.from_numpy(wp).to(dev)
    if args.w8:
        w_pre0 = wq.prepack_weight_w8(wd, wl.K, wl.N, wl.G)
    else:
        w_pre0 = wq.prepack_weight(wd, wl.K, wl.N, wl.G)
    del wd
    w_pre = [w_pre0] + [w_pre0.clone() for _ in range(copies - 1)]
    xs = [xd] + [xd.clone() for _ in range(copies - 1)]
    ss = [sd] + [sd.clone() for _ in range(copies - 1)]
    ys = [torch.empty((wl.M, wl.N), dtype=torch.float16, device=dev) for _ in range(copies)]
    if args.w8:
        ws = [torch.zeros(wq.wqbmm_workspace_bytes_w8(wl.M, wl.K, wl.N, wl.G), dtype=torch.uint8, device=dev)
              for _ in range(copies)]
    else:
        ws = [wq.allocate_workspace(wl.M, wl.K, wl.N, wl.G, dev) for _ in range(copies)]
    zs = [None] * copies
    if args.zero_point != "none":
        zd = torch.from_numpy(I.make_zero_point(wl, args.zero_point)).to(dev)
        zs = [zd] + [zd.clone() for _ in range(copies - 1)]
    bd = torch.from_numpy(I.make_bias(wl)).to(dev) if args.bias else None
    optionals = args.zero_point != "none" or args.bias
    variant = optionals or args.per_channel or args.w8           # not the captured kernels' workload
    stream = torch.cuda.Stream(device=dev)

    def step(i, s):
        c = i % copies
        if args.w8:
            wq.wqbmm_run_w8(xs[c], w_pre[c], ss[c], zs[c], bd, ys[c], wl.M, wl.K, wl.N, wl.G, ws[c], None, s)
        elif optionals:
            wq.wqbmm_run_ex(xs[c], w_pre[c], ss[c], zs[c], bd, ys[c], wl.M, wl.K, wl.N, wl.G, ws[c], None, s)
        else:
            wq.wqbmm_run(xs[c], w_pre[c], ss[c], ys[c], wl.M, wl.K, wl.N, wl.G, ws[c], None, s)

    # ---- warm-up (eager, also sets kernel attributes before any capture)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i, stream)
    torch.cuda.synchronize()
    if wq.wqbmm_read_device_status(stream=stream) != 0:
        raise SystemExit("device status error during warm-up")

    # ---- graphs: a chunk of steps, replayed; the remainder in a second graph
    chunk = min(args.steps, 4 * copies)
    graphs = {}

    def graph_for(n):
        if n not in graphs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    step(i, torch.cuda.current_stream())
            graphs[n] = g
        return graphs[n]

    full, rem = divmod(args.steps, chunk)
    g_full = graph_for(chunk)
    g_rem = graph_for(rem) if rem else None
    torch.cuda.synchronize()

    sampler = ClockSampler(nvsmi_id(torch, dev, local))
    sampler.start()
    # sustained phase: steady clocks and at least a second of clock samples around the timed region
    t_end = time.time() + args.sustain_s
    with torch.cuda.stream(stream):
        while time.time() < t_end:
            g_full.replay()
            stream.synchronize()

    start_ev, stop_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start_ev.record(stream)
        for _ in range(full):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        stop_ev.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    time.sleep(0.25)
    sampler.stop()
    ms_total = slowest_rank_ms(start_ev.elapsed_time(stop_ev), world, dev)
    ms_step = ms_total / args.steps
    status = wq.wqbmm_read_device_status(stream=stream)
    if status != 0:
        raise SystemExit(f"device status error {status:#x}")

    # ---- end to end through the C ABI with host buffers: pinned x in, pinned y out, every step
    x_host = torch.from_numpy(x).pin_memory()
    y_host = torch.empty((wl.M, wl.N), dtype=torch.float16).pin_memory()
    e2e_steps = max(20, min(args.steps, 500))
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
        e2e_s = (time.perf_counter() - t0) / e2e_steps

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    # every path runs an unfold pre-pass and then the main kernel
    launches_per_step = 2
    peaks, peak_kind = measured_peaks()
    # the optional inputs add their own bytes: zero points 2 (K/G) N, bias 2 N
    alg_bytes = (wl.algorithmic_bytes() + (2 * wl.groups * wl.N if args.zero_point != "none" else 0) +
                 (2 * wl.N if args.bias else 0) + (wl.K * wl.N // 2 if args.w8 else 0))
    if wl.M <= 16:
        hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
        achieved = alg_bytes / (ms_step * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                    "frac": achieved / hbm_peak, "traffic": None if variant else dram_traffic(wl.name),
                    "peak_source": f"{peak_kind} hbm_gbs",
                    "algorithmic_bytes_per_launch": alg_bytes}
    else:
        # E4M3 dense tensor peak = the measured bf16 peak x 2 (the nominal fp8 : bf16 ratio 4.5 : 2.25)
        bf16 = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
        achieved = wl.int8_equiv_ops() / (ms_step * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": 2 * bf16, "unit": "TFLOP/s",
                    "frac": achieved / (2 * bf16), "traffic": None if variant else dram_traffic(wl.name),
                    "peak_source": f"{peak_kind} bf16_tflops x 2 (e4m3)",
                    "algorithmic_flops_per_launch": wl.int8_equiv_ops()}
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
                   "l2": f"{copies} rotating input copies ({copies * per_copy / 2**20:.0f} MiB > 2x L2)",
                   "launch": f"CUDA graphs of {chunk} steps"},
        "gpu_launches": args.steps * launches_per_step,
        "clocks": sampler.summary(),
        "e2e": {"value": metric_value(wl, e2e_s, 1, args.w8), "unit": unit, "h2d_bytes_per_step": int(x.nbytes),
                "d2h_bytes_per_step": int(wl.M * wl.N * 2),
                "note": "eager wqbmm_run per step; pinned x in, pinned y out, stream synchronized each step"},
        "roofline": roofline,
    }
    if not args.no_cpu_baseline:
        v, cores, sample, dt = cpu_oracle_baseline(wl, args.cpu_baseline_s)
        line["cpu_baseline"] = {"value": v, "unit": unit, "cores": cores, "kind": "oracle", "sample": sample,
                                "s_per_call": dt}
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
