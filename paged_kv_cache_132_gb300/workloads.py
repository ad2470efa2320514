"""Seeded synthetic decode workloads, shared by the GPU path and the oracle.

This module only draws inputs: context lengths, block tables and slot numbers
(through the host block manager), and normally distributed payloads for the
KV pools, queries and new tokens.  It holds none of the attention arithmetic.

The five workloads stand in for the pages' evaluation workloads (which use
the ShareGPT/Alpaca/WMT16 datasets and OPT/LLaMA weights, none of which is
used here); their shapes follow the models the pages evaluate:

  tiny               4 seqs, ctx {5,17,33,64}, 4 heads (MHA), d 64, fp32, B 16,
                     32-block pool in a seeded random order.
  opt13b             64 seqs, 40 heads (MHA), d 128, fp16, B 16, ctx ~ U[128,2048],
                     pool 1.1x the blocks needed, random block order.
  llama8b            256 seqs, 32 query / 8 KV heads, d 128, bf16, B 16,
                     ctx = clip(round(LogNormal(ln 1024, 1.0)), 16, 8192),
                     pool = exactly the blocks needed, shuffled.
  parallel_sampling  32 prompts x 8 samples, llama8b head shape, bf16, B 16;
                     1000-token prompt shared through reference counts, tails
                     ~ U[0,512] per sample; copy-on-write of the partial last
                     prompt block (7 copies per prompt) before the tails are
                     written; pool 1.1x the blocks used, shuffled.
  long_context       16 seqs x 32768 ctx, llama8b head shape, bf16, shuffled,
                     512-token partitions; block size 8, 16 or 32 (same tokens).

Every workload describes one decode step: (1) the copy-on-write pairs (only
parallel_sampling has any), (2) the new tokens' K/V and their slots, (3) the
queries, with context lengths that include the token written in (2).  Slots
not holding a cached token are filled with NaN, so a kernel that lets a stale
slot reach its sums fails every comparison.

Payloads are drawn on ``device`` with a generator seeded from the workload's
seed; the integer structure (lengths, tables, slots) is always drawn on the
CPU, so it is identical for every device.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Dict, List, Optional

import torch

from .block_manager import BlockManager, blocks_needed

SEED_BASE = 132000

WORKLOADS = ("tiny", "opt13b", "llama8b", "parallel_sampling", "long_context")
_INDEX = {name: i for i, name in enumerate(WORKLOADS)}


@dataclass
class Workload:
    name: str
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: torch.dtype
    num_blocks: int
    scale: float
    partition_size: int              # 0: the library picks
    context_lens: torch.Tensor       # int32 [S], includes this step's token
    block_tables: torch.Tensor       # int32 [S][max_blocks], -1 past each table
    query: torch.Tensor              # [S][H][d]
    k_cache: torch.Tensor            # [NB][Hkv][B][d], before the step
    v_cache: torch.Tensor
    new_key: torch.Tensor            # [T][Hkv][d]
    new_value: torch.Tensor
    slot_mapping: torch.Tensor       # int64 [T]
    copy_pairs: torch.Tensor         # int64 [n][2] (src, dst)
    seed: int = 0
    notes: Dict[str, object] = field(default_factory=dict)

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max().item()) if self.num_seqs else 0

    @property
    def num_tokens(self) -> int:
        return int(self.slot_mapping.numel())

    def to(self, device) -> "Workload":
        moved = {}
        for f in ("context_lens", "block_tables", "query", "k_cache", "v_cache", "new_key",
                  "new_value", "slot_mapping", "copy_pairs"):
            moved[f] = getattr(self, f).to(device)
        return replace(self, **moved)


# ---------------------------------------------------------------------------
# integer structure
# ---------------------------------------------------------------------------
def _permutation(n: int, gen: torch.Generator) -> List[int]:
    return torch.randperm(n, generator=gen).tolist()


def _tables_tensor(tables: List[List[int]]) -> torch.Tensor:
    width = max([len(t) for t in tables] + [1])
    out = torch.full((len(tables), width), -1, dtype=torch.int32)
    for s, t in enumerate(tables):
        if t:
            out[s, : len(t)] = torch.tensor(t, dtype=torch.int32)
    return out


def _decode_step_structure(ctx: List[int], block_size: int, num_blocks: int, gen: torch.Generator):
    """Tables for sequences whose first ctx-1 tokens are cached, plus the slot
    of each sequence's new token (position ctx-1).  Sequences with ctx = 0
    have no token to write."""
    mgr = BlockManager(num_blocks, block_size, _permutation(num_blocks, gen))
    history_slots, new_slots = [], []
    for s, n in enumerate(ctx):
        mgr.add_sequence(s, max(n - 1, 0))
        history_slots.extend(mgr.prompt_slots(s))
        if n > 0:
            new_slots.append(mgr.append_token(s))
    tables = [mgr.table(s) for s in range(len(ctx))]
    return tables, history_slots, new_slots


# ---------------------------------------------------------------------------
# payloads
# ---------------------------------------------------------------------------
def _normal(shape, dtype, gen, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(dtype)


def _pool_from_tokens(tokens: torch.Tensor, slots: List[int], num_blocks: int, block_size: int) -> torch.Tensor:
    """Pool [NB][Hkv][B][d] holding token i's rows at slot slots[i], NaN elsewhere."""
    t, hkv, d = tokens.shape
    flat = torch.full((num_blocks * block_size, hkv, d), float("nan"), dtype=tokens.dtype,
                      device=tokens.device)
    if t:
        index = torch.tensor(slots, dtype=torch.int64, device=tokens.device)
        flat.index_copy_(0, index, tokens)
    return flat.view(num_blocks, block_size, hkv, d).permute(0, 2, 1, 3).contiguous()


def _assemble(name, ctx, tables, history_slots, new_slots, copy_pairs, *, num_heads, num_kv_heads,
              head_dim, block_size, dtype, num_blocks, partition_size, seed, device, notes=None):
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    n_hist = len(history_slots)
    keys = _normal((n_hist, num_kv_heads, head_dim), dtype, gen, device)
    values = _normal((n_hist, num_kv_heads, head_dim), dtype, gen, device)
    k_cache = _pool_from_tokens(keys, history_slots, num_blocks, block_size)
    del keys
    v_cache = _pool_from_tokens(values, history_slots, num_blocks, block_size)
    del values
    s = len(ctx)
    query = _normal((s, num_heads, head_dim), dtype, gen, device)
    t = len(new_slots)
    new_key = _normal((t, num_kv_heads, head_dim), dtype, gen, device)
    new_value = _normal((t, num_kv_heads, head_dim), dtype, gen, device)
    return Workload(
        name=name, num_seqs=s, num_heads=num_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
        block_size=block_size, dtype=dtype, num_blocks=num_blocks,
        scale=1.0 / math.sqrt(head_dim), partition_size=partition_size,
        context_lens=torch.tensor(ctx, dtype=torch.int32, device=device),
        block_tables=_tables_tensor(tables).to(device),
        query=query, k_cache=k_cache, v_cache=v_cache, new_key=new_key, new_value=new_value,
        slot_mapping=torch.tensor(new_slots, dtype=torch.int64, device=device),
        copy_pairs=torch.tensor(copy_pairs, dtype=torch.int64, device=device).reshape(-1, 2),
        seed=seed, notes=dict(notes or {}))


# ---------------------------------------------------------------------------
# the five workloads
# ---------------------------------------------------------------------------
def _simple(name, ctx, *, num_heads, num_kv_heads, head_dim, block_size, dtype, num_blocks,
            partition_size, seed, device, gen_cpu, notes=None):
    tables, hist, new = _decode_step_structure(ctx, block_size, num_blocks, gen_cpu)
    return _assemble(name, ctx, tables, hist, new, [], num_heads=num_heads,
                     num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=block_size,
                     dtype=dtype, num_blocks=num_blocks, partition_size=partition_size,
                     seed=seed, device=device, notes=notes)


def custom(ctx: List[int], *, num_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
           dtype: torch.dtype, num_blocks: Optional[int] = None, partition_size: int = 0,
           seed: int = SEED_BASE + 99, device="cpu", name="custom") -> Workload:
    """A decode step over arbitrary context lengths (edge cases, sweeps).
    The pool defaults to exactly the blocks needed, in a shuffled order."""
    gen_cpu = torch.Generator().manual_seed(seed)
    needed = sum(blocks_needed(n, block_size) for n in ctx)
    nb = max(num_blocks if num_blocks is not None else needed, 1)
    return _simple(name, list(ctx), num_heads=num_heads, num_kv_heads=num_kv_heads,
                   head_dim=head_dim, block_size=block_size, dtype=dtype, num_blocks=nb,
                   partition_size=partition_size, seed=seed, device=device, gen_cpu=gen_cpu)


def make(name: str, device="cpu", *, block_size: Optional[int] = None, num_seqs: Optional[int] = None,
         seed: Optional[int] = None) -> Workload:
    """Build workload ``name`` (see the module docstring).  ``num_seqs`` keeps
    only the first n sequences (a smaller case with the same distribution);
    ``block_size`` selects the long_context sweep point."""
    if name not in _INDEX:
        raise KeyError(f"unknown workload {name!r}; choose from {WORKLOADS}")
    seed = SEED_BASE + _INDEX[name] if seed is None else seed
    gen_cpu = torch.Generator().manual_seed(seed)

    if name == "tiny":
        ctx = [5, 17, 33, 64][: num_seqs or 4]
        return _simple(name, ctx, num_heads=4, num_kv_heads=4, head_dim=64, block_size=16,
                       dtype=torch.float32, num_blocks=32, partition_size=0, seed=seed,
                       device=device, gen_cpu=gen_cpu)

    if name == "opt13b":
        s = 64
        ctx = torch.randint(128, 2049, (s,), generator=gen_cpu).tolist()[: num_seqs or s]
        needed = sum(blocks_needed(n, 16) for n in ctx)
        return _simple(name, ctx, num_heads=40, num_kv_heads=40, head_dim=128, block_size=16,
                       dtype=torch.float16, num_blocks=math.ceil(1.1 * needed), partition_size=0,
                       seed=seed, device=device, gen_cpu=gen_cpu)

    if name == "llama8b":
        s = 256
        draw = torch.empty(s, dtype=torch.float64).log_normal_(math.log(1024.0), 1.0, generator=gen_cpu)
        ctx = torch.clamp(torch.round(draw), 16, 8192).to(torch.int64).tolist()[: num_seqs or s]
        needed = sum(blocks_needed(n, 16) for n in ctx)
        return _simple(name, ctx, num_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                       dtype=torch.bfloat16, num_blocks=needed, partition_size=0, seed=seed,
                       device=device, gen_cpu=gen_cpu,
                       notes={"lognormal": "mu=ln(1024), sigma=1.0, rounded, clipped to [16,8192]"})

    if name == "long_context":
        bs = block_size or 16
        if bs not in (8, 16, 32):
            raise ValueError("long_context sweeps block sizes 8, 16 and 32")
        s = num_seqs or 16
        ctx = [32768] * s
        # The token payload depends only on the seed, not on the block size,
        # so the three sweep points hold the same batch.
        needed = sum(blocks_needed(n, bs) for n in ctx)
        tables, hist, new = _decode_step_structure(ctx, bs, needed, gen_cpu)
        return _assemble(name, ctx, tables, hist, new, [], num_heads=32, num_kv_heads=8,
                         head_dim=128, block_size=bs, dtype=torch.bfloat16, num_blocks=needed,
                         partition_size=512, seed=seed, device=device)

    # parallel_sampling
    prompts, samples, prompt_len, bs = 32, 8, 1000, 16
    if num_seqs is not None:
        prompts = max(1, num_seqs // samples)
    tails = torch.randint(0, 513, (prompts * samples,), generator=gen_cpu).tolist()

    def simulate(num_blocks, free_order):
        mgr = BlockManager(num_blocks, bs, free_order)
        hist = []
        for p in range(prompts):
            base = p * samples
            mgr.add_sequence(base, prompt_len)
            hist.extend(mgr.prompt_slots(base))
            for i in range(1, samples):
                mgr.fork(base, base + i)
        new = []
        for seq in range(prompts * samples):
            for _ in range(tails[seq] + 1):  # the tail, then this step's token
                new.append(mgr.append_token(seq))
        used = num_blocks - mgr.num_free()
        return mgr, hist, new, used

    bound = prompts * samples * (blocks_needed(prompt_len + 513, bs) + 1)
    _, _, _, used = simulate(bound, None)
    nb = math.ceil(1.1 * used)
    mgr, hist, new, _ = simulate(nb, _permutation(nb, gen_cpu))
    pairs = mgr.take_copies()
    ctx = [prompt_len + tails[q] + 1 for q in range(prompts * samples)]
    tables = [mgr.table(q) for q in range(prompts * samples)]
    return _assemble(name, ctx, tables, hist, new, pairs, num_heads=32, num_kv_heads=8,
                     head_dim=128, block_size=bs, dtype=torch.bfloat16, num_blocks=nb,
                     partition_size=0, seed=seed, device=device,
                     notes={"prompts": prompts, "samples": samples, "prompt_len": prompt_len,
                            "unique_blocks_used": used})


# ---------------------------------------------------------------------------
# beam search: sharing that changes every step
# ---------------------------------------------------------------------------
@dataclass
class BeamStep:
    """One decode step of beam search: copy-on-write pairs, then the new
    tokens' K/V and slots, then attention for every live beam."""
    copy_pairs: torch.Tensor     # int64 [n][2]
    slot_mapping: torch.Tensor   # int64 [beams]
    new_key: torch.Tensor        # [beams][Hkv][d]
    new_value: torch.Tensor
    block_tables: torch.Tensor   # int32 [beams][max_blocks] after this step
    context_lens: torch.Tensor   # int32 [beams]
    query: torch.Tensor          # [beams][H][d]
    freed_blocks: int            # blocks returned to the pool at this step


@dataclass
class BeamSearchTrace:
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: torch.dtype
    num_blocks: int
    scale: float
    k_cache: torch.Tensor        # pool after the prompt, before step 0
    v_cache: torch.Tensor
    steps: List[BeamStep]


def beam_search(*, beams: int = 4, prompt_len: int = 45, steps: int = 40, num_heads: int = 8,
                num_kv_heads: int = 2, head_dim: int = 64, block_size: int = 4, dtype=torch.bfloat16,
                requests: int = 1, seed: int = SEED_BASE + 10, device="cpu") -> BeamSearchTrace:
    """A seeded beam-search trace ("PagedAttention 论文精读笔记", §6.2, Fig. 9).

    Each of `requests` prompts is stored once and shared by its beams.  At
    every step each of a request's `beams` new candidates picks a parent among
    that request's current beams (uniformly, with replacement): parents picked
    several times are forked (blocks shared, refcount + 1), beams not picked
    die and their blocks are released (freed when the count reaches zero).
    Every candidate then appends its token; a shared last block is first
    copied (copy-on-write).  Sequence r*beams + j is beam j of request r."""
    gen_cpu = torch.Generator().manual_seed(seed)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    per_beam = blocks_needed(prompt_len + steps + 1, block_size)
    num_blocks = requests * (blocks_needed(prompt_len, block_size) + beams * (per_beam + 2))
    mgr = BlockManager(num_blocks, block_size, _permutation(num_blocks, gen_cpu))
    prompt_slots = []
    live = []
    next_id = 0
    for _ in range(requests):
        mgr.add_sequence(next_id, prompt_len)
        prompt_slots.extend(mgr.prompt_slots(next_id))
        live.append([next_id])
        next_id += 1
    n = len(prompt_slots)
    keys = _normal((n, num_kv_heads, head_dim), dtype, gen, device)
    values = _normal((n, num_kv_heads, head_dim), dtype, gen, device)
    k_cache = _pool_from_tokens(keys, prompt_slots, num_blocks, block_size)
    v_cache = _pool_from_tokens(values, prompt_slots, num_blocks, block_size)
    del keys, values
    total = requests * beams
    out_steps = []
    for _ in range(steps):
        free_before = mgr.num_free()
        new_live = []
        for r in range(requests):
            parents = torch.randint(0, len(live[r]), (beams,), generator=gen_cpu).tolist()
            kids = []
            for p in parents:
                mgr.fork(live[r][p], next_id)
                kids.append(next_id)
                next_id += 1
            for seq in live[r]:
                mgr.free_sequence(seq)
            new_live.append(kids)
        freed = mgr.num_free() - free_before
        live = new_live
        seqs = [seq for kids in live for seq in kids]
        slots = [mgr.append_token(seq) for seq in seqs]
        pairs = mgr.take_copies()
        out_steps.append(BeamStep(
            copy_pairs=torch.tensor(pairs, dtype=torch.int64, device=device).reshape(-1, 2),
            slot_mapping=torch.tensor(slots, dtype=torch.int64, device=device),
            new_key=_normal((total, num_kv_heads, head_dim), dtype, gen, device),
            new_value=_normal((total, num_kv_heads, head_dim), dtype, gen, device),
            block_tables=_tables_tensor([mgr.table(seq) for seq in seqs]).to(device),
            context_lens=torch.tensor([mgr.length(seq) for seq in seqs], dtype=torch.int32, device=device),
            query=_normal((total, num_heads, head_dim), dtype, gen, device),
            freed_blocks=freed))
    return BeamSearchTrace(num_heads=num_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                           block_size=block_size, dtype=dtype, num_blocks=num_blocks,
                           scale=1.0 / math.sqrt(head_dim), k_cache=k_cache, v_cache=v_cache, steps=out_steps)


# ---------------------------------------------------------------------------
# prefill over a shared, cached prefix
# ---------------------------------------------------------------------------
@dataclass
class PrefillStep:
    """One prompt step over a cached prefix ("PagedAttention 论文精读笔记",
    §6.3): copy-on-write of the shared partial last prefix block, then the new
    tokens' K/V written to their slots, then attention of every new token over
    the prefix and the new tokens up to itself."""
    name: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: torch.dtype
    num_blocks: int
    scale: float
    k_cache: torch.Tensor          # [NB][Hkv][B][d]: the prefixes cached, NaN elsewhere
    v_cache: torch.Tensor
    copy_pairs: torch.Tensor       # int64 [n][2]
    new_key: torch.Tensor          # [T][Hkv][d], T = sum of the chunk lengths
    new_value: torch.Tensor
    slot_mapping: torch.Tensor     # int64 [T]
    query: torch.Tensor            # [T][H][d]
    query_start_loc: torch.Tensor  # int32 [S+1]
    context_lens: torch.Tensor     # int32 [S]: prefix + chunk
    block_tables: torch.Tensor     # int32 [S][max_blocks]
    max_query_len: int
    chunk_lens: List[int]
    prefix_lens: List[int]
    notes: Dict[str, object] = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return len(self.chunk_lens)

    @property
    def num_tokens(self) -> int:
        return int(self.query.shape[0])

    def attended_pairs(self) -> int:
        """(new token, position) pairs the step attends, per query head."""
        return sum(n * p + n * (n + 1) // 2 for n, p in zip(self.chunk_lens, self.prefix_lens))


PREFILL_WORKLOADS = ("prefill_tiny", "prefill_llama8b", "prefill_opt13b")


def prefill_custom(chunk_lens: List[int], prefix_lens: List[int], *, prefix_groups: Optional[List[int]] = None,
                   num_heads: int, num_kv_heads: int, head_dim: int, block_size: int, dtype: torch.dtype,
                   seed: int = SEED_BASE + 20, device="cpu", name="prefill_custom",
                   notes=None) -> PrefillStep:
    """Requests with chunk_lens[s] new tokens after a cached prefix.
    prefix_groups[s] names the prefix request s shares (default: its own);
    prefix_lens[g] is the length of prefix g.  Each prefix is stored once
    and forked into its requests (reference counts); a request's first new
    token copies the shared partial last block (copy-on-write)."""
    s_count = len(chunk_lens)
    groups = list(range(s_count)) if prefix_groups is None else list(prefix_groups)
    if len(groups) != s_count or any(g < 0 or g >= len(prefix_lens) for g in groups):
        raise ValueError("prefix_groups must name one prefix per request")
    gen_cpu = torch.Generator().manual_seed(seed)
    holders = [10 ** 7 + g for g in range(len(prefix_lens))]

    def simulate(num_blocks, free_order):
        mgr = BlockManager(num_blocks, block_size, free_order)
        hist = []
        for g, plen in enumerate(prefix_lens):
            mgr.add_sequence(holders[g], plen)
            hist.extend(mgr.prompt_slots(holders[g]))
        for s in range(s_count):
            mgr.fork(holders[groups[s]], s)
        new = []
        for s in range(s_count):
            for _ in range(chunk_lens[s]):
                new.append(mgr.append_token(s))
        return mgr, hist, new, num_blocks - mgr.num_free()

    bound = sum(blocks_needed(p, block_size) for p in prefix_lens) + sum(
        blocks_needed(prefix_lens[groups[s]] + chunk_lens[s], block_size) + 1 for s in range(s_count))
    _, _, _, used = simulate(max(bound, 1), None)
    nb = max(math.ceil(1.1 * used), 1)
    mgr, hist, new, _ = simulate(nb, _permutation(nb, gen_cpu))
    pairs = mgr.take_copies()
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    keys = _normal((len(hist), num_kv_heads, head_dim), dtype, gen, device)
    values = _normal((len(hist), num_kv_heads, head_dim), dtype, gen, device)
    k_cache = _pool_from_tokens(keys, hist, nb, block_size)
    v_cache = _pool_from_tokens(values, hist, nb, block_size)
    del keys, values
    t = len(new)
    starts = [0]
    for n in chunk_lens:
        starts.append(starts[-1] + n)
    per_seq_prefix = [prefix_lens[groups[s]] for s in range(s_count)]
    return PrefillStep(
        name=name, num_heads=num_heads, num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=block_size,
        dtype=dtype, num_blocks=nb, scale=1.0 / math.sqrt(head_dim), k_cache=k_cache, v_cache=v_cache,
        copy_pairs=torch.tensor(pairs, dtype=torch.int64, device=device).reshape(-1, 2),
        new_key=_normal((t, num_kv_heads, head_dim), dtype, gen, device),
        new_value=_normal((t, num_kv_heads, head_dim), dtype, gen, device),
        slot_mapping=torch.tensor(new, dtype=torch.int64, device=device),
        query=_normal((t, num_heads, head_dim), dtype, gen, device),
        query_start_loc=torch.tensor(starts, dtype=torch.int32, device=device),
        context_lens=torch.tensor([per_seq_prefix[s] + chunk_lens[s] for s in range(s_count)], dtype=torch.int32,
                                  device=device),
        block_tables=_tables_tensor([mgr.table(s) for s in range(s_count)]).to(device),
        max_query_len=max(chunk_lens + [0]), chunk_lens=list(chunk_lens), prefix_lens=per_seq_prefix,
        notes=dict(notes or {}, unique_blocks_used=used))


def make_prefill(name: str, device="cpu", *, num_seqs: Optional[int] = None,
                 seed: Optional[int] = None) -> PrefillStep:
    """The prefill workloads (stand-ins for the pages' shared-prefix
    translation workload, with a synthetic few-shot prefix; no dataset):

      prefill_tiny     3 requests, chunks {1, 50, 130} after one shared 37-token
                       prefix, 8 query / 2 KV heads, d 64, bf16, B 16.
      prefill_llama8b  32 requests sharing one 1024-token prefix, chunks
                       ~ U[128, 1024]; 32 query / 8 KV heads, d 128, bf16, B 16.
      prefill_opt13b   16 requests, 4 prefixes of 512 tokens (4 requests each),
                       chunks ~ U[128, 1024]; 40 heads (MHA), d 128, f16, B 16.
    """
    if name not in PREFILL_WORKLOADS:
        raise KeyError(f"unknown prefill workload {name!r}; choose from {PREFILL_WORKLOADS}")
    seed = SEED_BASE + 30 + PREFILL_WORKLOADS.index(name) if seed is None else seed
    gen_cpu = torch.Generator().manual_seed(seed)
    if name == "prefill_tiny":
        chunks = [1, 50, 130][: num_seqs or 3]
        return prefill_custom(chunks, [37], prefix_groups=[0] * len(chunks), num_heads=8, num_kv_heads=2,
                              head_dim=64, block_size=16, dtype=torch.bfloat16, seed=seed, device=device,
                              name=name)
    if name == "prefill_llama8b":
        s = num_seqs or 32
        chunks = torch.randint(128, 1025, (32,), generator=gen_cpu).tolist()[:s]
        return prefill_custom(chunks, [1024], prefix_groups=[0] * s, num_heads=32, num_kv_heads=8, head_dim=128,
                              block_size=16, dtype=torch.bfloat16, seed=seed, device=device, name=name,
                              notes={"chunks": "U[128,1024]", "prefix": 1024})
    s = num_seqs or 16
    chunks = torch.randint(128, 1025, (16,), generator=gen_cpu).tolist()[:s]
    return prefill_custom(chunks, [512] * 4, prefix_groups=[i % 4 for i in range(s)], num_heads=40,
                          num_kv_heads=40, head_dim=128, block_size=16, dtype=torch.float16, seed=seed,
                          device=device, name=name, notes={"chunks": "U[128,1024]", "prefix": "4 x 512"})
