"""The benchmark's multi-rank host logic with two gloo ranks on the CPU.

bench.py runs one independent replica per GPU (the MSA forward shards by
(sequence, KV head, query tile) with no exchange step); the only cross-rank
operations are a barrier and the max over ranks of the step time. This runs
those with world_size 2 on the gloo backend, no GPU involved.
"""
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


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        assert (w, r, local) == (world, rank, rank)
        bench.barrier(world)
        # Rank r's step took (r + 1) * 10 ms: the job's time is the slowest rank's.
        t = bench.max_over_ranks(0.010 * (rank + 1), world)
        value = bench.aggregate_value(4.0e12, world, t)
        results[rank] = (t, value)
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    mp.start_processes(_rank_main, args=(world, port, results), nprocs=world, join=True,
                       start_method="spawn")
    for rank in range(world):
        t, value = results[rank]
        assert t == pytest.approx(0.020)
        # Whole-job throughput: both replicas' work over the slowest rank's time.
        assert value == pytest.approx(2 * 4.0e12 / 0.020)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(0.5, 1) == 0.5
    assert bench.aggregate_value(10.0, 1, 2.0) == 5.0
