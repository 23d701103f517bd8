"""The N-GPU bench path runs replicas: each rank does the same step on its own
GPU, the job time is the slowest rank's, and the value is the work of all
ranks over that time. The rank logic is exercised here on CPU with gloo at
world size 2 (no GPU involved)."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [3.0, 5.5][rank]                       # this rank's step time (ms)
        worst = bench.reduce_max(mine, world, "cpu")
        value = bench.job_throughput(2.0e12, world, worst * 1e-3)
        out.put((rank, worst, value))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_with_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(out.get(timeout=10) for _ in range(world))
    for rank, worst, value in got:
        assert worst == 5.5                             # every rank sees the slowest
        assert value == pytest.approx(2 * 2.0e12 / 5.5e-3 / 1e12)


def test_single_rank_is_identity():
    assert bench.reduce_max(1.25, 1, "cpu") == 1.25
    assert bench.job_throughput(1.0e12, 1, 0.5) == pytest.approx(2.0)


def test_reference_arm_runs_on_rank_zero_only():
    class A:
        steps, warmup = 1, 0
    assert bench.reference_arm(A(), rank=1, world=2) is None
