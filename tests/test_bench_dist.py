"""The N>1 host logic of bench.py on CPU: two gloo ranks, barrier, max- and
sum-over-ranks (the whole-job value is all ranks' work / the slowest rank)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, local, w = bench.dist_env()
    assert (r, local, w) == (rank, rank, world)
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    t = bench.max_over_ranks(10.0 + rank, w)
    units = bench.sum_over_ranks(100.0 * (rank + 1), w)
    out[rank] = (t, units)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1] == (11.0, 300.0)
