"""Head-sharded decode on the CPU: the oracle per shard, concatenated, is the
unsharded oracle, bit for bit ("PagedAttention 论文精读笔记", §8.1 and §8.2:
every worker holds the same block ids but only its heads' K/V, and attention
needs no collective).  One test runs two gloo ranks that receive the step's
block tables from the scheduler rank, compute their heads and gather the
output."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from paged_kv_cache_132_gb300 import sharding, workloads
from steps import oracle_decode, oracle_pools


def _oracle_step(w):
    k, v = oracle_pools(w)
    return oracle_decode(w, k, v)


def test_head_ranges():
    assert sharding.kv_head_range(8, 4, 0) == (0, 2)
    assert sharding.kv_head_range(8, 4, 3) == (6, 8)
    assert sharding.query_head_range(32, 8, 4, 1) == (8, 16)
    assert sharding.query_head_range(40, 40, 8, 7) == (35, 40)
    with pytest.raises(ValueError):
        sharding.kv_head_range(8, 3, 0)
    with pytest.raises(ValueError):
        sharding.kv_head_range(8, 2, 2)


def test_shard_keeps_block_ids_and_heads():
    w = workloads.make("tiny", device="cpu")
    s = sharding.shard_workload(w, 2, 1)
    assert s.k_cache.shape == (w.num_blocks, 2, w.block_size, w.head_dim)
    assert torch.equal(s.k_cache.view(torch.int32), w.k_cache[:, 2:4].contiguous().view(torch.int32))
    assert torch.equal(s.query, w.query[:, 2:4])
    assert torch.equal(s.new_value, w.new_value[:, 2:4])
    assert s.block_tables is w.block_tables and s.slot_mapping is w.slot_mapping
    assert (s.num_heads, s.num_kv_heads) == (2, 2)


@pytest.mark.parametrize("name,kw,worlds", [
    ("llama8b", {"num_seqs": 6}, (2, 4, 8)),
    ("opt13b", {"num_seqs": 3}, (2, 5, 8)),
    ("parallel_sampling", {"num_seqs": 16}, (2, 8)),
    ("tiny", {}, (2, 4)),
])
def test_oracle_shards_concatenate_to_the_unsharded_output(name, kw, worlds):
    w = workloads.make(name, device="cpu", **kw)
    full = _oracle_step(w)
    for world in worlds:
        parts = [_oracle_step(sharding.shard_workload(w, world, r)) for r in range(world)]
        got = np.concatenate(parts, axis=1)
        assert np.array_equal(got, full), f"{name}: {world} shards differ from the unsharded oracle"


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = workloads.make("parallel_sampling", device="cpu", num_seqs=16)
        if rank != 0:
            # workers hold no memory-management state: the scheduler's tables arrive by broadcast
            w = workloads.Workload(**{**w.__dict__, "block_tables": torch.zeros_like(w.block_tables),
                                      "context_lens": torch.zeros_like(w.context_lens),
                                      "slot_mapping": torch.zeros_like(w.slot_mapping),
                                      "copy_pairs": torch.zeros_like(w.copy_pairs)})
        w = sharding.broadcast_control(w, src=0)
        local = torch.from_numpy(_oracle_step(sharding.shard_workload(w, world, rank)))
        out = sharding.gather_heads(local, world)
        results[rank] = out.numpy().tobytes()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_gather_the_unsharded_output():
    world = 2
    manager = mp.get_context("spawn").Manager()
    results = manager.dict()
    mp.spawn(_worker, args=(world, _free_port(), results), nprocs=world, join=True)
    full = _oracle_step(workloads.make("parallel_sampling", device="cpu", num_seqs=16))
    for rank in range(world):
        got = np.frombuffer(results[rank], dtype=np.float64).reshape(full.shape)
        assert np.array_equal(got, full), f"rank {rank}'s gathered output differs from the unsharded oracle"
