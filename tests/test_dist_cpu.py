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


def _heads_worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        args = bench.parse_args(["--split", "heads", "--workload", "llama8b", "--num-seqs", "6"])
        w = bench.make_workload(args, rank, world, device="cpu")
        # every rank holds its KV heads of the same batch: same tables, its query heads
        from paged_kv_cache_132_gb300 import sharding
        q = sharding.gather_heads(w.query.float(), world)
        cfg = bench.decode_config(args, w, world, 512, 0, (w.num_heads * world, w.num_kv_heads * world))
        results[rank] = (w.num_heads, w.num_kv_heads, w.block_tables.tolist(), q.numpy().tobytes(), cfg)
    finally:
        dist.destroy_process_group()


def test_two_rank_head_split_of_the_bench():
    """bench.py --split heads on two gloo ranks: each rank keeps half of the
    KV heads (and their query heads) of the one batch, with the same block
    tables; the gathered queries are the whole batch's; both ranks describe
    the same job (the batch's full head counts, tp2)."""
    world = 2
    manager = mp.get_context("spawn").Manager()
    results = manager.dict()
    mp.spawn(_heads_worker, args=(world, _free_port(), results), nprocs=world, join=True)
    full = bench.make_workload(bench.parse_args(["--workload", "llama8b", "--num-seqs", "6"]), 0, 1, device="cpu")
    (h0, hk0, t0, q0, c0), (h1, hk1, t1, q1, c1) = results[0], results[1]
    assert (h0, hk0) == (h1, hk1) == (16, 4)
    assert t0 == t1 == full.block_tables.tolist()
    import numpy as np
    assert np.array_equal(np.frombuffer(q0, dtype=np.float32).reshape(full.query.shape), full.query.float().numpy())
    assert q0 == q1
    assert c0 == c1 and "32 query / 8 KV heads" in c0["workload"] and c0["parallelism"].startswith("tp2")
