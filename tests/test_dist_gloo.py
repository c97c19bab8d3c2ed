"""The benchmark's multi-rank bookkeeping (replicas, barrier, max over ranks) on CPU with gloo, world size 2."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    d = bench.Dist()
    d.barrier()
    local_secs = 1.0 + rank          # rank 1 is the slow one
    worst = d.max(local_secs)
    rate = bench.aggregate_rate([100] * world, [worst] * world)
    q.put((rank, worst, rate))
    d.close()


def test_two_rank_max_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks agree on the slowest rank's time; whole-job rate = all units over that time
    assert [r[1] for r in res] == [2.0, 2.0]
    assert [r[2] for r in res] == [100.0, 100.0]


def test_aggregate_rate_single():
    import bench
    assert bench.aggregate_rate([50], [0.5]) == 100.0
    assert bench.aggregate_rate([10, 10, 10], [1.0, 2.0, 4.0]) == pytest.approx(7.5)


def test_popular_experts_order():
    """Hot-set choice from expert offsets: chunks with rows first, then rows, then the lower id."""
    import bench
    # 3 chunks, 5 experts: rows per (chunk, expert)
    rows = [[0, 4, 1, 0, 2],
            [3, 0, 1, 0, 2],
            [0, 0, 1, 7, 0]]
    offs = [[0] + list(__import__("itertools").accumulate(r)) for r in rows]
    # chunks with rows: e0 1, e1 1, e2 3, e3 1, e4 2; rows: e0 3, e1 4, e2 3, e3 7, e4 4
    assert bench.popular_experts(offs, 5) == [2, 4, 3, 1, 0]
    assert bench.popular_experts(offs, 2) == [2, 4]
    assert bench.popular_experts(offs, 0) == []
