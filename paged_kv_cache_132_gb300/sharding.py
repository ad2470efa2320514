"""Head-sharded decode: the KV cache and the attention of one layer split by
KV head over the ranks of a tensor-parallel group.

"PagedAttention 论文精读笔记", §8.1 (tensor parallelism) and §8.2 (distributed
KV cache management): every worker runs the same scheduler decisions, so all
of them hold the same block tables and slot numbers, while each stores, in
its own physical blocks of those ids, only the K/V of the attention heads it
owns.  Attention is independent per head, so a worker computes its heads'
outputs from its own memory alone and needs no collective inside attention;
the all-reduce of a tensor-parallel layer comes after the output projection,
which is not part of this path.

Here rank r of N owns the contiguous KV heads [r * Hkv/N, (r+1) * Hkv/N) and
with them the query heads of their GQA groups, [r * H/N, (r+1) * H/N) (query
head h reads KV head h / G, G = H / Hkv, so a contiguous range of KV heads
carries a contiguous range of query heads).  A rank's pools are
[NB][Hkv/N][B][d]: the same block ids as the unsharded pools, each block
holding only the rank's heads.  Its cache write takes the rank's heads of the
new tokens with the same slots; its decode is the unchanged pa_decode with
num_heads = H/N and num_kv_heads = Hkv/N on the same tables and lengths.  The
layer's output [S][H][d] is the concatenation of the ranks' outputs along the
head axis, in rank order.

This module only slices inputs and concatenates outputs (torch tensor views
and copies); every step of the path still runs in the library's kernels.
"""
from __future__ import annotations

from dataclasses import replace
from typing import List, Optional, Sequence, Tuple

import torch

from .workloads import Workload


def kv_head_range(num_kv_heads: int, world: int, rank: int) -> Tuple[int, int]:
    """[lo, hi) of the KV heads rank `rank` of `world` owns."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a group of {world}")
    if num_kv_heads % world:
        raise ValueError(f"{num_kv_heads} KV heads do not split evenly over {world} ranks")
    per = num_kv_heads // world
    return rank * per, (rank + 1) * per


def query_head_range(num_heads: int, num_kv_heads: int, world: int, rank: int) -> Tuple[int, int]:
    """[lo, hi) of the query heads that go with the rank's KV heads."""
    if num_heads % num_kv_heads:
        raise ValueError("num_heads must be a multiple of num_kv_heads")
    group = num_heads // num_kv_heads
    lo, hi = kv_head_range(num_kv_heads, world, rank)
    return lo * group, hi * group


def shard_pool(pool: torch.Tensor, world: int, rank: int) -> torch.Tensor:
    """The rank's pool [NB][Hkv/N][B][d] (a contiguous copy) of a pool
    [NB][Hkv][B][d]: the same block ids, the rank's heads only."""
    lo, hi = kv_head_range(pool.shape[1], world, rank)
    return pool[:, lo:hi].contiguous()


def shard_tokens(rows: torch.Tensor, world: int, rank: int) -> torch.Tensor:
    """The rank's heads of new tokens' K or V, [T][Hkv][d] -> [T][Hkv/N][d]."""
    lo, hi = kv_head_range(rows.shape[1], world, rank)
    return rows[:, lo:hi].contiguous()


def shard_query(query: torch.Tensor, num_kv_heads: int, world: int, rank: int) -> torch.Tensor:
    """The rank's query heads, [S][H][d] -> [S][H/N][d]."""
    lo, hi = query_head_range(query.shape[1], num_kv_heads, world, rank)
    return query[:, lo:hi].contiguous()


def shard_workload(w: Workload, world: int, rank: int) -> Workload:
    """Rank `rank`'s part of a decode step: its heads of the pools, the
    queries and the new tokens; the same tables, lengths, slots and
    copy-on-write pairs (block ids are shared by every rank)."""
    if world == 1:
        return w
    return replace(
        w, num_heads=w.num_heads // world, num_kv_heads=w.num_kv_heads // world,
        query=shard_query(w.query, w.num_kv_heads, world, rank),
        k_cache=shard_pool(w.k_cache, world, rank), v_cache=shard_pool(w.v_cache, world, rank),
        new_key=shard_tokens(w.new_key, world, rank), new_value=shard_tokens(w.new_value, world, rank),
        notes={**w.notes, "head_shard": (rank, world)})


def concat_heads(outputs: Sequence[torch.Tensor]) -> torch.Tensor:
    """The layer's output [S][H][d] from the ranks' outputs [S][H/N][d], in
    rank order."""
    return torch.cat(list(outputs), dim=1)


def gather_heads(local_out: torch.Tensor, world: int, group: Optional[object] = None) -> torch.Tensor:
    """All ranks' outputs concatenated along the head axis, on every rank
    (torch.distributed.all_gather).  Attention itself needs no exchange;
    this assembles the full output where a caller wants it in one place (a
    check, or a layer whose next step is not tensor-parallel)."""
    if world == 1:
        return local_out
    import torch.distributed as dist

    parts: List[torch.Tensor] = [torch.empty_like(local_out) for _ in range(world)]
    dist.all_gather(parts, local_out.contiguous(), group=group)
    return concat_heads(parts)


def broadcast_control(w: Workload, src: int = 0, group: Optional[object] = None) -> Workload:
    """The step's memory-management inputs -- block tables, context lengths,
    slots of the new tokens, copy-on-write pairs -- sent from the scheduler's
    rank `src` to every rank ("PagedAttention 论文精读笔记", §8.2: the
    scheduler broadcasts each step's block tables with the step's inputs;
    workers keep no memory-management state of their own).  Every rank must
    pass tensors of the same shapes; the received values replace its own."""
    import torch.distributed as dist

    fields = ("block_tables", "context_lens", "slot_mapping", "copy_pairs")
    got = {}
    for name in fields:
        t = getattr(w, name).contiguous().clone()
        dist.broadcast(t, src=src, group=group)
        got[name] = t
    return replace(w, **got)
