"""The multi-rank path of bench.py on CPU: two gloo ranks on 127.0.0.1.

The layer shards by rows with no exchange (rows are independent and the
reduction tree never depends on M), so the only cross-rank operations are the
timing barrier and the reductions of the step time (max over ranks) and of the
work done (sum over ranks)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    try:
        d.barrier()
        t = d.max(1.0 + rank)            # slowest rank's time
        f = d.sum(10.0 * (rank + 1))     # work of all ranks
        rows = bench.shard_rows(1000, world, rank)
        q.put((rank, t, f, rows, d.world))
    finally:
        d.close()


def test_two_gloo_ranks_reduce_time_and_work():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, t, f, rows, w in res:
        assert w == 2 and t == 2.0 and f == 30.0
    # rows are split into disjoint contiguous ranges that cover everything
    (r0, r1) = res[0][3], res[1][3]
    assert r0[0] == 0 and r0[1] == r1[0] and r1[1] == 1000


def test_shard_rows_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.shard_rows(17, 1, 0) == (0, 17)
    spans = [bench.shard_rows(17, 4, r) for r in range(4)]
    assert spans[0][0] == 0 and spans[-1][1] == 17
    assert all(spans[i][1] == spans[i + 1][0] for i in range(3))
