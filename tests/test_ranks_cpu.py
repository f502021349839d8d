"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

Each GPU runs an independent replica of the workload (the path needs no
inter-GPU exchange), so the only cross-rank steps are a barrier and the max of
the per-rank step times; the whole-job throughput counts every rank's tokens
within the slowest rank's time.  These tests run those steps as two gloo
processes on 127.0.0.1 and check the results, and that the reference arm
leaves ranks other than 0 without work.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.ranks_barrier(world)
        slowest = bench.ranks_max(times[rank], world, "cpu")
        out[rank] = (slowest, bench.job_throughput(slowest, 32768, world))
        bench.ranks_barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_every_rank():
    world, port = 2, _free_port()
    times = [4.0, 5.0]  # ms per step of each replica
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        slowest, value = res[r]
        assert slowest == 5.0
        assert value == pytest.approx(2 * 32768 / 5e-3)


def test_single_rank_is_a_no_op():
    sys.path.insert(0, ROOT)
    import bench
    bench.ranks_barrier(1)
    assert bench.ranks_max(3.5, 1, "cpu") == 3.5
    assert bench.job_throughput(2.0, 1000, 1) == pytest.approx(5e5)


def test_reference_arm_does_no_work_off_rank_zero(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    called = []
    monkeypatch.setattr(bench, "oracle_sample", lambda *a, **k: called.append(1))
    assert bench.run_reference(type("A", (), {"workload": "stateful32k", "T": 0,
                                              "warmup": 1, "steps": 1, "gpus": 2})()) == 0
    assert not called
