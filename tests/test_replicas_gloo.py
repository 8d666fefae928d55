"""The multi-GPU path is independent replicas: the only cross-rank step is the
host-side aggregation of the timing (slowest rank's time, all ranks' bytes).
Checked with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t, b = bench.aggregate(1.5 + rank, 1000 * (rank + 1), dist, "cpu")
        q.put((rank, t, b))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, b in res:
        assert t == 2.5          # the slower rank's step time
        assert b == 3000.0       # both ranks' bytes


def test_single_process_aggregation_is_identity():
    assert bench.aggregate(0.7, 123) == (0.7, 123.0)
