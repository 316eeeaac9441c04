"""The N > 1 path of bench.py on CPU: two gloo ranks, each timing its own
replica; the job's time is the slowest rank's and the rate counts the units
of every rank."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.replica_max(times[rank], world, "cpu")
        out[rank] = (ms, bench.replica_rate(1048576, ms, world))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_rate():
    pytest.importorskip("torch.distributed")
    world, port = 2, _free_port()
    times = [0.25, 0.31]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        ms, rate = res[r]
        assert ms == max(times)
        assert rate == pytest.approx(world * 1048576 / (max(times) * 1e-3))


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.replica_max(0.5, 1, "cpu") == 0.5
    assert bench.replica_rate(100, 2.0, 1) == pytest.approx(5e4)
