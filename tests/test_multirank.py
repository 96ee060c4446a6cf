"""The multi-rank path of bench.py on CPU ranks (gloo, world size 2): each
rank runs its own batch of the same shape, the reported time is the slowest
rank's, and throughput counts every rank's tokens."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from harness import WORKLOADS
    w = bench.replica_workload(WORKLOADS["titans_mlp"], rank)
    slowest = bench.max_over_ranks(1.0 + rank)          # rank r "took" 1 + r seconds
    out[rank] = (w.seed, w.tokens, slowest, bench.job_throughput(w.tokens, world, 3, slowest))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    (s0, n0, t0, v0), (s1, n1, t1, v1) = out[0], out[1]
    assert s0 != s1 and n0 == n1                       # distinct batches, same shape
    assert t0 == t1 == 2.0                              # both ranks see the slowest time
    assert v0 == v1 == pytest.approx(n0 * world * 3 / 2.0)
