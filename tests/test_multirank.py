"""The benchmark's multi-rank logic on CPU ranks (gloo, world size 2): every rank runs its own
replica, the job is timed by the slowest rank, and the rate counts every rank's units."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(dist, times[rank], "cpu")
        out[rank] = (ms, bench.whole_job_rate(1000.0, world, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_slowest_rank_times_the_job_and_rate_counts_all_ranks():
    world, times = 2, [3.0, 5.0]
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, _free_port(), times, out), nprocs=world, join=True)
    for rank in range(world):
        ms, rate = out[rank]
        assert ms == pytest.approx(5.0)
        assert rate == pytest.approx(1000.0 * world / 5e-3)


def test_single_process_needs_no_collective():
    assert bench.max_over_ranks(None, 4.0, "cpu") == 4.0
    assert bench.whole_job_rate(10.0, 1, 2.0) == pytest.approx(5000.0)


def test_reference_arm_does_nothing_on_nonzero_ranks(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    args = bench.argparse.Namespace(steps=1, warmup=0, cpu_seconds=0.1)
    bench.run_reference(args)
    assert capsys.readouterr().out == ""
