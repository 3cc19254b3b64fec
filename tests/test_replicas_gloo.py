"""Multi-GPU path on CPU: bench.py runs N independent replicas (the layer has
no exchange step on one GPU) and reports the whole job's throughput against
the slowest rank.  Two gloo ranks check the reduction and the aggregate."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)

    def max_over_ranks(v):
        t = torch.tensor([v], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    local_ms = 2.0 + rank          # rank 1 is the slow one
    tps, ms = bench.replica_throughput(local_ms, 128, world, max_over_ranks)
    out[rank] = (tps, ms)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_replicas_report_the_slowest_rank():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        tps, ms = out[r]
        assert ms == 3.0                               # max over ranks
        assert tps == pytest.approx(world * 128 / 3e-3)


def test_single_rank_is_identity():
    tps, ms = bench.replica_throughput(2.0, 128, 1, None)
    assert ms == 2.0 and tps == pytest.approx(64000.0)
