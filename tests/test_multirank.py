"""The N > 1 host path of bench.py on CPU: two gloo ranks, each a replica
with its own step time; the job's time is the slowest rank's and the
throughput counts every rank's bytes (no GPU, no data-path collective)."""
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


def _rank(rank, world, port, times, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], world, torch.device("cpu"))
        out[rank] = (ms, bench.job_gbs(1_000_000, ms, world))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_sum_bytes():
    world, times = 2, [0.5, 0.8]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), times, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        ms, gbs = res[r]
        assert ms == pytest.approx(0.8)
        assert gbs == pytest.approx(2 * 1_000_000 / 0.8e-3 / 1e9)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(1.25, 1, torch.device("cpu")) == 1.25
    assert bench.job_gbs(2_000_000, 2.0, 1) == pytest.approx(1.0)
