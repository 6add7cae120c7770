"""Multi-rank logic of bench.py on CPU: two gloo ranks on 127.0.0.1.

Each rank converts its own weight in a multi-GPU run (weak scaling, no data
collective); the ranks meet only in barriers and one MAX all-reduce of the
elapsed time, and only rank 0 prints.  Those pieces are exercised here
without a GPU."""

import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import argparse

    import torch.distributed as dist

    import bench

    r, w = bench.dist_env()
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    slowest = bench.max_over_ranks(10.0 + 5.0 * rank, w)
    # the reference arm: only rank 0 works and prints, the others return at once
    args = argparse.Namespace(steps=1, warmup=0, gpus=w)
    ref = bench.run_reference(args, r, w) if r != 0 else "skipped-on-rank-0"
    bench.barrier(w)
    dist.destroy_process_group()
    q.put((r, w, slowest, ref))


def test_two_gloo_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(rank, 2, port, q)) for rank in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    assert [o[0] for o in out] == [0, 1]
    assert all(o[1] == 2 for o in out)
    assert all(o[2] == pytest.approx(15.0) for o in out)  # max over ranks
    assert out[1][3] is None  # rank 1 of the reference arm does no work


def test_single_rank_needs_no_process_group():
    import sys

    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
