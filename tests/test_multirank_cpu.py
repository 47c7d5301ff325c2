"""The multi-GPU path is replicas only: each rank runs its own batch and the
only cross-rank step is the harness's barrier and max-over-ranks timing.
This checks that step with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    times = [3.5, 7.25]
    slowest = bench.max_over_ranks(times[rank], world)
    seeds = [bench.replica_seed(0, r) for r in range(world)]
    out[rank] = (slowest, seeds[rank], len(set(seeds)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_distinct_workloads():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                           join=True, start_method="spawn")
        res = dict(out)
    assert res[0][0] == pytest.approx(7.25) and res[1][0] == pytest.approx(7.25)
    assert res[0][1] != res[1][1] and res[0][2] == world
