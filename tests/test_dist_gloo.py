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
