"""bench.py's multi-rank bookkeeping on CPU: two gloo ranks (replicas) agree
on the job clock (the slowest rank's time) and on the whole-job value."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + 5.0 * rank  # rank 1 is the slow one
        job_ms = bench.max_over_ranks(torch, mine, dist, torch.device("cpu"))
        dist.barrier()
        out[rank] = (job_ms, bench.job_tflops(world, 8.0e12, job_ms))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_share_the_slowest_clock():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert sorted(res) == [0, 1]
    for rank in range(world):
        job_ms, value = res[rank]
        assert job_ms == 15.0
        # two replicas of an 8 TFLOP step in 15 ms: 2 * 8e12 / 15e-3 / 1e12
        assert value == pytest.approx(2 * 8.0e12 / 15e-3 / 1e12)


def test_single_process_clock_is_its_own():
    torch = pytest.importorskip("torch")
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(torch, 12.5, None, None) == 12.5
    assert bench.job_tflops(1, 8.0e12, 10.0) == pytest.approx(800.0)
