"""The bench's multi-rank logic on CPU with two gloo ranks: the step time is
the maximum over ranks, and the reference arm does its work on rank 0 only
(the other ranks return without work and print nothing)."""
import os
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        mine = [0.25, 1.75][rank]                       # this rank's ms per step
        got = bench.max_over_ranks(mine, torch.device("cpu"), world)
        # rank 0 would run minutes of oracle work; only the other ranks are checked here
        ref = bench.run_reference(None, rank, world) if rank != 0 else "skipped"
        q.put((rank, got, ref))
    finally:
        torch.distributed.destroy_process_group()


def test_max_over_ranks_and_reference_rank_gloo():
    world, port = 2, 29517
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [1.75, 1.75]          # every rank sees the slowest rank's time
    assert res[1][2] is None                             # rank 1 does no reference work


def test_max_over_ranks_single_process():
    import bench
    assert bench.max_over_ranks(3.5, torch.device("cpu"), 1) == 3.5
