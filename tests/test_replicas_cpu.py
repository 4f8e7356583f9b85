"""The benchmark's multi-GPU plumbing (replicas only: every rank runs an independent canvas pass,
no data-path collective) on two CPU ranks over gloo: the barrier, the max-over-ranks timing and
the whole-job aggregate."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    bench.init_dist(ws, "gloo")
    bench.barrier(ws)
    # rank r "took" 1.5 + r seconds for 10 canvas passes
    t = bench.max_over_ranks(1.5 + rank, ws, torch.device("cpu"))
    value = bench.aggregate(10, t, ws)
    out.put((rank, t, value))
    bench.barrier(ws)
    dist.destroy_process_group()


def test_two_rank_replica_timing_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, value in res:
        assert t == pytest.approx(2.5)          # the slowest rank's time, seen by every rank
        assert value == pytest.approx(20 / 2.5)  # all ranks' passes over that time


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.0, 1, torch.device("cpu")) == 3.0
    assert bench.aggregate(7, 2.0, 1) == 3.5
