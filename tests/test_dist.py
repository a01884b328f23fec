"""World-size-2 gloo check (CPU) of the bench's replica aggregation: every
rank times its own replica; the job value is the sum of the ranks' work over
the slowest rank's time."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r = bench.Ranks()
    r.barrier()
    t = r.max(1.0 + rank)            # rank 1 is slower
    work = r.sum(10.0 * (rank + 1))  # 10 + 20 units
    out[rank] = (r.rank, r.world, t, work, work / t)
    r.close()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(i, 2, port, out)) for i in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] or (out[0][2:] == out[1][2:])
    rank, world, t, work, value = out[0]
    assert world == 2 and t == 2.0 and work == 30.0 and value == 15.0


def test_single_rank_is_identity():
    for k in ("RANK", "WORLD_SIZE"):
        os.environ.pop(k, None)
    import bench
    r = bench.Ranks()
    assert r.world == 1 and r.max(3.5) == 3.5 and r.sum(2.0) == 2.0
