"""World-size-2 gloo check (CPU) of the replica aggregation bench.py uses for N > 1:
whole-job throughput = units summed over ranks / the slowest rank's time."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    d = bench.Dist()
    d.init("gloo")
    units = 100.0 * (rank + 1)          # ranks did different amounts of work
    secs = 0.5 + rank                   # rank 1 is the slowest
    v, tmax = bench.aggregate(units, secs, d)
    d.barrier()
    q.put((rank, v, tmax))
    d.close()


def test_replica_aggregation_world2():
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
    for _, v, tmax in res:
        assert tmax == pytest.approx(1.5)
        assert v == pytest.approx(300.0 / 1.5)


def test_single_rank_aggregation_is_identity():
    import bench

    d = bench.Dist()
    assert d.world == int(os.environ.get("WORLD_SIZE", 1))
    if d.world == 1:
        assert bench.aggregate(10.0, 2.0, d) == (5.0, 2.0)
