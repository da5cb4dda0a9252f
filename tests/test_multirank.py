"""The benchmark's multi-rank path on CPU, with two gloo ranks.

The path has no exchange of its own (replicas only): `bench.py --gpus N` runs
one full batch per rank and the only collective is the reduction of the timer,
the slowest rank's time, from which the whole-job rate counts every rank's
requests. These tests run that reduction and the rate in two spawned gloo
processes, and check that the reference arm does no work on ranks other than 0.
"""
from __future__ import annotations

import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [12.5, 20.0, 7.0, 9.0][rank]
    got = bench.max_over_ranks(ms, torch, dist, world, torch.device("cpu"))
    rate = bench.whole_job_rate(world, 32, 10, got)
    dist.barrier()
    q.put((rank, got, rate))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_timer_reduction_and_rate_over_gloo_ranks(world):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    slowest = max([12.5, 20.0, 7.0, 9.0][:world])
    for rank, got, rate in results:
        assert got == slowest
        assert rate == pytest.approx(world * 32 * 10 / (slowest / 1000.0))


def test_single_rank_needs_no_process_group():
    import torch
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, torch, None, 1, torch.device("cpu")) == 3.25
    assert bench.whole_job_rate(1, 32, 20, 10.0) == pytest.approx(64000.0)


def test_reference_arm_is_rank0_only(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        gpus, steps, warmup = 2, 1, 1
    bench.run_reference(Args(), rank=1)
    assert capsys.readouterr().out == ""
