"""The bench's multi-rank logic (independent replicas, one per GPU under
torchrun) on CPU: two gloo ranks, no GPU.  The replicas share nothing but
the barrier and the max-over-ranks step time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, step_ms, flops, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        dist.barrier()
        slowest = bench.max_over_ranks(step_ms[rank], ws, torch.device("cpu"))
        value = bench.job_tflops(flops, slowest, ws)
        dist.barrier()
        out.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_take_the_slowest_rank():
    ws = 2
    step_ms = [2.0, 3.0]                 # rank 1 is the slower replica
    flops = 2 * 4096 ** 3
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, step_ms, flops, out))
             for r in range(ws)]
    for p in procs:
        p.start()
    results = [out.get(timeout=120) for _ in range(ws)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value in results:
        assert slowest == 3.0
        # ws replicas' FLOPs over the slowest rank's time
        assert value == pytest.approx(ws * flops / 3e-3 / 1e12)


def test_single_rank_is_the_identity():
    assert bench.max_over_ranks(2.5, 1, torch.device("cpu")) == 2.5
    assert bench.job_tflops(2e12, 1000.0, 1) == pytest.approx(2.0)


def test_reference_arm_runs_on_rank_zero_only():
    class Args:
        workloads = ["f32_256"]
        cpu_seconds = 0.1
        steps = 1
        warmup = 0
    assert bench.run_reference(Args(), 2, 1) is None
