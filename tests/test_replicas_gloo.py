"""The N>1 path on CPU: independent replicas, one per rank (world_size 2,
gloo), aggregated with the max step time over ranks (weak scaling)."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r pretends its replica took 100 + 50 r ms for 1e15 flops
    value, ms = bench.aggregate_throughput(100.0 + 50.0 * rank, 1e15, world)
    out[rank] = (value, ms, bench.max_over_ranks(float(rank), world))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        value, ms, mx = out[r]
        assert ms == 150.0                       # max over ranks
        assert abs(value - 2 * 1e15 / 0.150 / 1e12) < 1e-6  # whole-job aggregate
        assert mx == 1.0


def test_single_rank_is_identity():
    import bench
    value, ms = bench.aggregate_throughput(200.0, 1e15, 1)
    assert ms == 200.0 and abs(value - 5000.0) < 1e-9
