"""The multi-process path of the benchmark on CPU (gloo, world size 2).

Each rank of a torchrun launch runs its own replica of the workload (the path
shards into independent sequences with no exchange); the job's time is the
slowest rank's, and the whole-job throughput counts every rank's bytes.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from paged_kv_cache_132_gb300 import workloads


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        # each rank draws its own replica: same shapes, different lengths and payloads
        seed = workloads.SEED_BASE + 2 + 1000 * rank
        w = workloads.make("llama8b", device="cpu", num_seqs=8, seed=seed)
        step_ms = 1.0 + rank  # rank 1 is the slower one
        slowest = bench.all_reduce_max(step_ms, world, device="cpu")
        bench.barrier(world)
        results[rank] = (slowest, w.context_lens.tolist(), w.num_seqs)
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_take_the_slowest_time():
    world = 2
    # the manager process is spawned too: forking a process that already
    # runs threads can deadlock the child
    manager = mp.get_context("spawn").Manager()
    results = manager.dict()
    mp.spawn(_worker, args=(world, _free_port(), results), nprocs=world, join=True)
    (slow0, ctx0, n0), (slow1, ctx1, n1) = results[0], results[1]
    assert slow0 == slow1 == 2.0
    assert n0 == n1 == 8 and ctx0 != ctx1
    # whole-job throughput: both ranks' bytes over the slowest rank's time
    assert bench.aggregate_throughput(world, 1e9, 2.0) == pytest.approx(1000.0)
    assert bench.aggregate_throughput(1, 1e9, 1.0) == pytest.approx(1000.0)
