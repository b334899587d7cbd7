"""The N > 1 path of the benchmark's host logic on CPU: two gloo ranks, each
with its own time; every rank gets the slowest rank's time, and the whole-job
rate counts the bytes of both ranks against it (replicas, no data exchange)."""
import datetime
import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=60))
    try:
        ms = [2.5, 3.25][rank]                       # rank 1 is the slower one
        got = bench.reduce_max(ms, world, "cpu")
        out[rank] = (got, bench.job_rate(7_568_097_280, world, got))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert res[0][0] == res[1][0] == 3.25
    assert res[0][1] == res[1][1]
    assert abs(res[0][1] - 2 * 7_568_097_280 / 3.25e-3 / 1e9) < 1e-9 * res[0][1]


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(1.5, 1, "cpu") == 1.5
    assert abs(bench.job_rate(1e9, 1, 1.0) - 1000.0) < 1e-9
