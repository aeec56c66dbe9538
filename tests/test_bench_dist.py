"""The bench's multi-rank plumbing on CPU: two gloo ranks.

With N ranks the bench runs N independent replicas; whole-job throughput is
the units all ranks processed divided by the slowest rank's time.  These
tests run that host logic (barrier, sum, max) in two spawned processes.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    d = bench.Dist(backend="gloo")
    d.barrier()
    value, t = bench.aggregate(d, per_rank_units=float(rank + 1), per_rank_seconds=0.5 * (rank + 1))
    q.put((rank, value, t, d.world, d.rank))
    d.close()


@pytest.mark.timeout(120)
def test_two_rank_aggregate_uses_sum_of_units_over_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=90)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, value, t, world, r in res:
        assert world == 2 and r == rank
        assert t == pytest.approx(1.0)            # the slowest rank's time
        assert value == pytest.approx(3.0)        # (1 + 2) units / 1.0 s


def test_single_rank_aggregate_is_local():
    import bench
    d = bench.Dist()
    assert d.world == int(os.environ.get("WORLD_SIZE", "1"))
    value, t = bench.aggregate(d, 6.0, 2.0) if d.world == 1 else (3.0, 2.0)
    assert value == pytest.approx(3.0) and t == pytest.approx(2.0)
