"""Multi-GPU runs are independent replicas: no data-path collective, only the
timing reduction (the slowest replica) and the whole-job per-token value.  The
cross-rank logic of bench.py runs here as two gloo ranks on the CPU."""
from __future__ import annotations

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_setup()
        mine = [10.0 + 5.0 * rank, 3.0 - rank, 7.0]   # per-rank timings (ms)
        got = bench.max_over_ranks(mine, dist, "cpu")
        value = bench.per_token_us(got[0], steps=3, tokens_per_step=1024, world=w)
        q.put((r, w, local, got, value))
    finally:
        dist.destroy_process_group()


def test_two_replicas_reduce_to_the_slowest():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, w, local, got, value) in enumerate(res):
        assert (rank, w, local) == (r, world, r)
        assert got == [15.0, 3.0, 7.0]   # element-wise max over the ranks
        # slowest replica's 15 ms over 2 ranks x 3 steps x 1024 tokens
        assert value == pytest.approx(15.0e3 / (3 * 1024 * 2))


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2.5], None, "cpu") == [1.5, 2.5]
    assert bench.per_token_us(30.0, 30, 1024, 1) == pytest.approx(30.0e3 / (30 * 1024))
