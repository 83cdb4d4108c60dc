"""The bench's multi-rank host logic with world size 2 over gloo on CPU: the
barrier, the max over ranks, and the whole-job throughput (units of every
rank over the slowest rank's time).  N > 1 runs are independent replicas; the
only exchange is this timing reduction."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    slowest = bench.max_over_ranks(10.0 * (rank + 1), world)
    # rank r took 100*(r+1) ms for 4 steps of 1e12 units
    thr = bench.job_throughput(1e12, 4, 100.0 * (rank + 1), world)
    bench.barrier(world)
    out[rank] = (slowest, thr)
    dist.destroy_process_group()


def test_two_rank_timing_reduction():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        slowest, thr = res[rank]
        assert slowest == 20.0
        # 2 ranks x 4 steps x 1e12 units over the slowest rank's 0.2 s
        assert abs(thr - 2 * 4 * 1e12 / 0.2) < 1e-3 * thr
