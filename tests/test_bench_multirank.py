"""The multi-rank (torchrun) aggregation of bench.py on CPU: world size 2 over gloo.

Each rank reports its own timed-region total and FLOPs; the job's time is the slowest rank's
and its value counts every rank's work.  No GPU is used.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    total_ms = [30.0, 50.0][rank]        # rank 1 is the slow one
    flops = [1.0e12, 1.5e12][rank]
    ms, value = bench.aggregate(total_ms, flops, steps=10, world=world, device=torch.device("cpu"))
    q.put((rank, ms, value))
    dist.destroy_process_group()


def test_aggregate_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, ms, value in res:
        assert ms == pytest.approx(5.0)                       # max(30, 50) ms / 10 steps
        assert value == pytest.approx(2.5e12 / 5e-3 / 1e12)   # both ranks' FLOPs / slowest time


def test_aggregate_single_rank():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    ms, value = bench.aggregate(20.0, 2.0e12, steps=4, world=1)
    assert ms == pytest.approx(5.0) and value == pytest.approx(400.0)
