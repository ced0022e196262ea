"""The multi-rank host logic of bench.py on CPU: two gloo ranks (127.0.0.1) agree on the
slowest rank's time and on the whole-job throughput, and under torchrun the reference arm
runs on rank 0 only (the other ranks return at once, printing nothing)."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(100.0 + 7.0 * rank, dist, torch.device("cpu"))
        gbs = bench.job_gbs(64 << 20, 10, world, slowest)
        dist.barrier()
        q.put((rank, slowest, gbs))
    finally:
        dist.destroy_process_group()


def test_two_ranks_agree_on_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [107.0, 107.0]
    want = 2 * (64 << 20) * 10 / 0.107 / 1e9
    assert all(abs(r[2] - want) < 1e-9 * want for r in res)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    class A:
        steps, warmup = 1, 0
    assert bench.reference_arm(A(), rank=1, world=2) == 0
    assert capsys.readouterr().out == ""


def test_job_gbs_is_weak_scaling_aggregate():
    one = bench.job_gbs(1 << 30, 5, 1, 10.0)
    assert bench.job_gbs(1 << 30, 5, 4, 10.0) == pytest.approx(4 * one)
