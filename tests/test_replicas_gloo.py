"""Multi-process (replica) host logic of bench.py on CPU: two gloo ranks, no GPU."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, local_ms, steps, out):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        dist.barrier()
        t, v = bench.job_throughput(world, steps, local_ms[rank], torch.device("cpu"))
        out[rank] = (t, v)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("local_ms", [(10.0, 25.0), (40.0, 8.0)])
def test_job_rate_uses_the_slowest_replica(local_ms):
    world, steps = 2, 50
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(world, _free_port(), local_ms, steps, out), nprocs=world,
                           start_method="spawn", join=True)
        res = dict(out)
    slow = max(local_ms)
    for rank in range(world):
        t, v = res[rank]
        assert t == slow                                       # every rank reports the max
        assert v == pytest.approx(world * steps / (slow * 1e-3))


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    t, v = bench.job_throughput(1, 20, 5.0, torch.device("cpu"))
    assert t == 5.0 and v == pytest.approx(4000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import argparse

    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = argparse.Namespace(workload="c1_tiny_f32_greedy", steps=3, warmup=3)
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""
