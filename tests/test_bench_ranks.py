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


def test_reference_arm_json_contract():
    # the reference arm (the oracle on the host cores) prints one JSON line with the keys the
    # benchmark contract names; one bounded step keeps this to tens of seconds
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                       cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert "workload" in line["config"]
