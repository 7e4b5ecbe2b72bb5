"""The benchmark's multi-rank path on CPU: two gloo ranks, barrier and max-over-ranks timing.

Each GPU runs an independent replica (one KV head per GPU, no exchange inside attention), so the only
cross-rank steps are the barrier and the reduction of the timed region to the slowest rank."""
import os
import socket

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import bench
    d = bench.Dist()
    d.barrier()
    seconds = 1.0 + rank          # rank 1 is the slow one
    value, t = bench.aggregate(per_rank_units=10.0, per_rank_seconds=seconds, dist=d)
    out[rank] = (value, t, d.world, d.rank)
    d.close()


def test_two_ranks_aggregate_over_the_slowest():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        value, t, world, rank = out[r]
        assert world == 2 and rank == r
        assert t == 2.0                      # max over ranks
        assert value == 10.0 * 2 / 2.0       # all ranks' units over the slowest rank's time


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(k, None)
    import bench
    d = bench.Dist()
    assert d.world == 1 and d.pg is None
    value, t = bench.aggregate(5.0, 2.5, d)
    assert (value, t) == (2.0, 2.5)
