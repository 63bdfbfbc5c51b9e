"""bench.py's multi-process host logic (replicas, max over ranks) on CPU with gloo."""
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


def _rank(rank, world, port, times, out):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = bench.max_over_ranks(times[rank], world)
        out[rank] = ms
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_gloo(world):
    times = [3.5, 7.25]
    out = mp.Manager().dict()
    port = _free_port()
    mp.spawn(_rank, args=(world, port, times, out), nprocs=world, join=True)
    assert [out[r] for r in range(world)] == [max(times)] * world  # every rank sees the slowest
    # whole-job value: the units of all ranks over the slowest rank's time
    assert bench.job_value(world, 4, max(times)) == pytest.approx(world * 4 * 1000.0 / 7.25)


def test_single_process_is_identity():
    assert bench.max_over_ranks(1.25, 1) == 1.25
    assert bench.job_value(1, 1, 8.0) == pytest.approx(125.0)
