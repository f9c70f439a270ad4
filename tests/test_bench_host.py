"""Host-side logic of bench.py: the metric arithmetic and the multi-rank (replica) timing reduction.

The replicas path runs here as two gloo ranks on the CPU: every rank reports its own timed-region length and all
must agree on the slowest one; the whole-job value scales with the number of replicas (weak scaling).
"""
import os
import socket

import pytest

import bench
from weight_quantized_matmul_gb300 import inputs as I

torch = pytest.importorskip("torch")


def test_metric_units_and_weak_scaling():
    dec = I.WORKLOADS["decode_m1_k4096_n4096"]
    assert bench.metric_for(dec)[1] == "GB/s"
    assert bench.units_per_step(dec) == 4096 * 4096 // 2
    assert bench.metric_value(dec, 1e-3) == pytest.approx(4096 * 4096 / 2 / 1e-3 / 1e9)
    pre = I.WORKLOADS["prefill_m2048_k8192_n28672"]
    assert bench.metric_for(pre)[1] == "TOPS"
    assert bench.units_per_step(pre) == 6 * 2048 * 8192 * 28672
    # N replicas each doing one step in the same time: N times the whole-job throughput
    assert bench.metric_value(pre, 2e-3, n=4) == pytest.approx(4 * bench.metric_value(pre, 2e-3))


def test_single_rank_time_is_its_own():
    assert bench.slowest_rank_ms(1.25, 1) == 1.25


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, _ = bench.dist_env()
        dist.barrier()
        q.put((r, w, bench.slowest_rank_ms(1.0 + 2.5 * r, w)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 2, 3.5), (1, 2, 3.5)]
