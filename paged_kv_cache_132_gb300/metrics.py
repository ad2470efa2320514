"""Byte counts used by the benchmark's roofline and by the capacity checks.

KV bytes per token: "paged-attention은 도대체 뭘 최적화 하는 것일까" (§ on the
size of the KV cache) and "PagedAttention 论文精读笔记", §3.1: one token stores a
key and a value vector per layer, so
    bytes/token = 2 x layers x (kv_heads x head_dim) x bytes per element
(OPT-13B: 2 x 40 x 5120 x 2 = 819,200 B, the pages' "800 KB").

Algorithmic bytes of one decode call: the K and V rows of exactly the tokens
attended (block padding and stale slots are not counted), plus the queries
read and the outputs written.  Block-table and context-length bytes are
reported separately.
"""
from __future__ import annotations

from typing import Iterable


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    return 2 * num_layers * num_kv_heads * head_dim * elem_bytes


def kv_token_capacity(cache_bytes: int, num_layers: int, num_kv_heads: int, head_dim: int,
                      elem_bytes: int) -> int:
    """Token slots that fit in ``cache_bytes`` of KV cache."""
    return cache_bytes // kv_bytes_per_token(num_layers, num_kv_heads, head_dim, elem_bytes)


def decode_kv_bytes(context_lens: Iterable[int], num_kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    return sum(int(n) for n in context_lens) * num_kv_heads * head_dim * 2 * elem_bytes


def decode_bytes(context_lens, num_heads: int, num_kv_heads: int, head_dim: int, elem_bytes: int,
                 out_elem_bytes: int) -> int:
    ctx = [int(n) for n in context_lens]
    s = len(ctx)
    return (decode_kv_bytes(ctx, num_kv_heads, head_dim, elem_bytes)
            + s * num_heads * head_dim * elem_bytes
            + s * num_heads * head_dim * out_elem_bytes)


def table_bytes(context_lens, block_size: int) -> int:
    ctx = [int(n) for n in context_lens]
    return sum((n + block_size - 1) // block_size for n in ctx) * 4 + 4 * len(ctx)


def write_bytes(num_tokens: int, num_kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    """Read new K/V, write them into the pools, read the slot numbers."""
    return 2 * 2 * num_tokens * num_kv_heads * head_dim * elem_bytes + 8 * num_tokens


def copy_bytes(num_pairs: int, num_layers: int, num_kv_heads: int, block_size: int, head_dim: int,
               elem_bytes: int) -> int:
    """Read + write of the K and V block of every pair and layer."""
    return 2 * 2 * num_pairs * num_layers * num_kv_heads * block_size * head_dim * elem_bytes


def prefill_flops(attended_pairs: int, num_heads: int, head_dim: int) -> int:
    """Useful flops of prefill attention: for every (query head, new token,
    attended position) pair, 2 d for q.k and 2 d for the weighted sum of v
    (positions the causal mask excludes are not counted)."""
    return 4 * head_dim * num_heads * int(attended_pairs)


def prefill_bytes(num_tokens: int, num_heads: int, kv_positions: int, num_kv_heads: int, head_dim: int,
                  elem_bytes: int, out_bytes: int) -> int:
    """Compulsory bytes of one prefill call: the queries, the outputs and each
    distinct K/V row read once (kv_positions = distinct cached positions)."""
    return num_tokens * num_heads * head_dim * (elem_bytes + out_bytes) + \
        2 * kv_positions * num_kv_heads * head_dim * elem_bytes
