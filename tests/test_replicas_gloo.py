"""The N>1 path on CPU: independent replicas, one per rank (world_size 2,
gloo), aggregated with the max step time over ranks (weak scaling).  Each
rank loads the library and builds its own plan of the bench workload; the
host-side results must agree across ranks."""

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
    from branch_attention_speculative_gb300 import api, workloads as W
    # every replica plans the same workload in its own process
    plan = api.Plan.from_workload(W.config(5))
    plan.validate()
    info = plan.info()
    digest = torch.tensor([float(info["main_pairs"]), float(info["workspace_bytes"]),
                           float(plan.table("bwd_kvtiles").sum())], dtype=torch.float64)
    gathered = [torch.zeros_like(digest) for _ in range(world)]
    dist.all_gather(gathered, digest)
    # rank r pretends its replica took 100 + 50 r ms for the plan's flops
    flops = info["fwd_flops"] + info["bwd_flops"]
    value, ms = bench.aggregate_throughput(100.0 + 50.0 * rank, flops, world)
    out[rank] = (value, ms, bench.max_over_ranks(float(rank), world), flops,
                 all(torch.equal(g, gathered[0]) for g in gathered))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    from branch_attention_speculative_gb300 import build as B
    B.build()  # once, before the ranks load it
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        value, ms, mx, flops, same = out[r]
        assert same                              # identical plans on every rank
        assert ms == 150.0                       # max over ranks
        assert abs(value - 2 * flops / 0.150 / 1e12) < 1e-6 * value  # whole-job aggregate
        assert mx == 1.0


def test_single_rank_is_identity():
    import bench
    value, ms = bench.aggregate_throughput(200.0, 1e15, 1)
    assert ms == 200.0 and abs(value - 5000.0) < 1e-9
