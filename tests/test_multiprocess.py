"""The benchmark's multi-rank host logic on CPU: two gloo ranks agree on the
slowest rank's time, the job rate counts every replica's work, and the
reference arm runs on rank 0 only."""
from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, ws: int, port: int, out):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        local_ms = 10.0 + 5.0 * rank                  # rank 1 is the slow one
        slowest = bench.max_over_ranks(local_ms, ws)
        rate = bench.job_rate(7.0e12, ws, slowest)
        dist.barrier()
        out.put((rank, slowest, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_count_all_work():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(ws))
    for rank, slowest, rate in got:
        assert slowest == 15.0
        assert rate == pytest.approx(2 * 7.0e12 / 15.0e-3)


def test_single_rank_is_a_no_op():
    import bench

    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.job_rate(1.0e12, 1, 500.0) == pytest.approx(2.0e12)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import bench

    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    class Args:
        workload, steps, warmup = "70b-layer", 1, 0

    # rank 1 returns before generating or timing anything
    assert bench.run_reference(Args()) == 0
