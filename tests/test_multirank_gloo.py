"""The benchmark's multi-rank plumbing on CPU: world size 2 over gloo.

The step runs as independent replicas, one per GPU; the only cross-rank
work is the timing reduction (max of times, sum of work) and the barriers
around the timed region.  Ranks are processes here, no GPU involved.
"""
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


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    assert bench.dist_env() == (world, rank, rank)
    bench.barrier()
    ms, units = bench.reduce_over_ranks(10.0 + 5.0 * rank, 3.0 + rank)
    out[rank] = (ms, units)
    bench.barrier()
    dist.destroy_process_group()


def test_reduce_over_ranks_two_gloo_ranks():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    # every rank sees the slowest rank's time and the work of all ranks
    assert res[0] == (15.0, 7.0) and res[1] == (15.0, 7.0)


def test_reduce_without_process_group_is_identity():
    import bench
    assert bench.reduce_over_ranks(3.5, 2.0) == (3.5, 2.0)
