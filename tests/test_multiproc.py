"""The multi-rank host logic of bench.py on CPU: two gloo ranks, each timing
its own replica; the job's time is the max over ranks and its work the sum."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_env()
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    elapsed = 10.0 + 5.0 * r           # rank 1 is the slow one
    work = 100.0 * (r + 1)
    q.put((r, bench.reduce_max(elapsed, w), bench.reduce_sum(work, w)))
    torch.distributed.destroy_process_group()


def test_two_rank_reduction():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 15.0, 300.0), (1, 15.0, 300.0)]


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5 and bench.reduce_sum(2.0, 1) == 2.0
