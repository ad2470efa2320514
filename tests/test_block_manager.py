"""Host block manager and workload generator (CPU only)."""
import math

import pytest
import torch

from paged_kv_cache_132_gb300 import workloads
from paged_kv_cache_132_gb300.block_manager import BlockManager, OutOfBlocks, blocks_needed


def test_blocks_needed_and_edges():
    assert blocks_needed(0, 16) == 0
    assert blocks_needed(1, 16) == 1
    assert blocks_needed(16, 16) == 1
    assert blocks_needed(17, 16) == 2
    with pytest.raises(ValueError):
        blocks_needed(-1, 16)


def test_refcounts_fork_and_free():
    mgr = BlockManager(10, 4)
    mgr.add_sequence(0, 6)            # blocks 0, 1
    mgr.fork(0, 1)
    assert mgr.refcount[0] == 2 and mgr.refcount[1] == 2
    slot = mgr.append_token(1)        # shared partial block 1 -> copy
    assert mgr.take_copies() == [(1, 2)]
    assert slot == 2 * 4 + 2
    assert mgr.refcount[1] == 1 and mgr.refcount[2] == 1
    slot0 = mgr.append_token(0)       # sole holder now: in place
    assert slot0 == 1 * 4 + 2 and mgr.take_copies() == []
    mgr.free_sequence(0)
    assert mgr.refcount[0] == 1 and mgr.refcount[1] == 0
    mgr.free_sequence(1)
    assert all(c == 0 for c in mgr.refcount)
    assert mgr.num_free() == 10


def test_out_of_blocks():
    mgr = BlockManager(2, 4)
    mgr.add_sequence(0, 8)
    with pytest.raises(OutOfBlocks):
        mgr.append_token(0)


def test_full_block_fork_needs_no_copy():
    mgr = BlockManager(8, 4)
    mgr.add_sequence(0, 8)            # two full blocks
    mgr.fork(0, 1)
    mgr.append_token(1)               # new block, no copy
    assert mgr.take_copies() == []


def test_tiny_workload_structure():
    w = workloads.make("tiny")
    assert w.context_lens.tolist() == [5, 17, 33, 64]
    assert w.num_blocks == 32
    used = w.block_tables[w.block_tables >= 0].tolist()
    assert len(used) == 1 + 2 + 3 + 4 and len(set(used)) == len(used)
    # new tokens at positions ctx-1: offsets 4, 0, 0, 15 in their blocks
    offs = [int(s) % 16 for s in w.slot_mapping.tolist()]
    assert offs == [4, 0, 0, 15]
    blocks = [int(s) // 16 for s in w.slot_mapping.tolist()]
    assert blocks == [int(w.block_tables[i, (n - 1) // 16]) for i, n in enumerate([5, 17, 33, 64])]


def test_parallel_sampling_structure():
    w = workloads.make("parallel_sampling", num_seqs=16)
    n = w.num_seqs
    prompts = n // 8
    assert w.copy_pairs.shape == (7 * prompts, 2)
    # every copy duplicates the partial last prompt block (logical block 62)
    tables = w.block_tables
    srcs = set(w.copy_pairs[:, 0].tolist())
    assert srcs == {int(tables[8 * p + 7, 62]) for p in range(prompts)}
    # the prefix blocks 0..61 are shared by all samples of a prompt
    for p in range(prompts):
        rows = tables[8 * p: 8 * p + 8, :62]
        assert torch.all(rows == rows[0])
    assert w.num_tokens == int((w.context_lens - 1000).sum())


def test_llama_lengths_distribution():
    g = torch.Generator().manual_seed(workloads.SEED_BASE + 2)
    draw = torch.empty(256, dtype=torch.float64).log_normal_(math.log(1024.0), 1.0, generator=g)
    ctx = torch.clamp(torch.round(draw), 16, 8192)
    assert 600 < float(ctx.median()) < 1700
    assert ctx.min() >= 16 and ctx.max() <= 8192


def test_beam_search_trace_bookkeeping():
    t = workloads.beam_search(beams=4, prompt_len=45, steps=40, block_size=4)
    b = t.block_size
    prev_tables = None
    total_copies = 0
    for i, st in enumerate(t.steps):
        ctx = st.context_lens.tolist()
        assert ctx == [45 + i + 1] * 4
        slots = st.slot_mapping.tolist()
        assert len(set(slots)) == len(slots), "two beams write the same slot"
        tables = st.block_tables
        for beam, slot in enumerate(slots):
            pos = ctx[beam] - 1
            assert slot == int(tables[beam, pos // b]) * b + pos % b
        pairs = st.copy_pairs.tolist()
        total_copies += len(pairs)
        dsts = [d for _, d in pairs]
        assert len(set(dsts)) == len(dsts)
        assert not set(dsts) & {s for s, _ in pairs}
        if prev_tables is not None:
            # a copied block was shared by the previous step's beams
            prev_blocks = set(prev_tables[prev_tables >= 0].tolist())
            assert all(src in prev_blocks for src, _ in pairs)
        prev_tables = tables
    assert total_copies > 0 and sum(st.freed_blocks for st in t.steps) > 0
