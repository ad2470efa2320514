"""Host-side KV block manager: the bookkeeping that produces the kernels' inputs.

It keeps a free list of physical blocks, one block table per sequence, a
reference count per physical block, and turns "append a token to sequence s"
into a slot number ``physical_block * block_size + offset`` -- the form in
which ``pa_reshape_and_cache`` takes a token's destination.

Sources:
  * "paged-attention은 도대체 뭘 최적화 하는 것일까", §5 (block table), §6
    (blocks taken from the free pool only when the last block is full), §17
    (ensure_capacity / write_kv), §18 step 8 (blocks return to the pool).
  * "PagedAttention 论文精读笔记", §5.3 (Fig. 6 decode walk-through), §6.1
    (reference counts and block-granular copy-on-write: a writer whose last
    block has refcount > 1 takes a new block, copies, and decrements; the last
    holder writes in place), §6.2 (beam search: blocks shared by several
    candidates, freed when the count drops to zero).

This is harness code (it builds inputs and copy lists on the host); the GPU
path never calls back into it.
"""
from __future__ import annotations

from collections import deque
from typing import Dict, Iterable, List, Optional, Tuple


def blocks_needed(num_tokens: int, block_size: int) -> int:
    """Blocks that hold ``num_tokens`` tokens: ceil(n / B)."""
    if num_tokens < 0 or block_size <= 0:
        raise ValueError("num_tokens must be >= 0 and block_size > 0")
    return (num_tokens + block_size - 1) // block_size


def wasted_slots(num_tokens: int, block_size: int) -> int:
    """Unused slots in a sequence's last block (at most block_size - 1)."""
    return blocks_needed(num_tokens, block_size) * block_size - num_tokens


class OutOfBlocks(RuntimeError):
    pass


class BlockManager:
    """Free list + block tables + reference counts + copy-on-write."""

    def __init__(self, num_blocks: int, block_size: int, free_order: Optional[Iterable[int]] = None):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = num_blocks
        self.block_size = block_size
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(order) != sorted(set(order)) or any(b < 0 or b >= num_blocks for b in order):
            raise ValueError("free_order must list distinct block ids in [0, num_blocks)")
        self.free: deque = deque(order)
        self.refcount: List[int] = [0] * num_blocks
        self.tables: Dict[int, List[int]] = {}
        self.lengths: Dict[int, int] = {}
        self.copies: List[Tuple[int, int]] = []  # (src, dst) pairs not yet handed out

    # -- allocation ---------------------------------------------------------
    def _allocate(self) -> int:
        if not self.free:
            raise OutOfBlocks("no free physical block")
        block = self.free.popleft()
        self.refcount[block] = 1
        return block

    def _release(self, block: int) -> None:
        self.refcount[block] -= 1
        if self.refcount[block] < 0:
            raise AssertionError(f"refcount of block {block} went negative")
        if self.refcount[block] == 0:
            self.free.append(block)

    # -- sequences ----------------------------------------------------------
    def add_sequence(self, seq_id: int, num_tokens: int) -> List[int]:
        """A new sequence whose first ``num_tokens`` tokens (its prompt) are
        stored now: takes ceil(n/B) blocks from the free list, in order."""
        if seq_id in self.tables:
            raise ValueError(f"sequence {seq_id} exists")
        self.tables[seq_id] = [self._allocate() for _ in range(blocks_needed(num_tokens, self.block_size))]
        self.lengths[seq_id] = num_tokens
        return list(self.tables[seq_id])

    def prompt_slots(self, seq_id: int) -> List[int]:
        """Slot numbers of positions 0..length-1 of a sequence."""
        return [self.slot(seq_id, pos) for pos in range(self.lengths[seq_id])]

    def fork(self, parent: int, child: int) -> None:
        """The child shares every block of the parent (refcount + 1 each)."""
        if child in self.tables:
            raise ValueError(f"sequence {child} exists")
        self.tables[child] = list(self.tables[parent])
        self.lengths[child] = self.lengths[parent]
        for block in self.tables[child]:
            self.refcount[block] += 1

    def slot(self, seq_id: int, position: int) -> int:
        """Slot of an already stored position: table[pos // B] * B + pos % B."""
        table = self.tables[seq_id]
        return table[position // self.block_size] * self.block_size + position % self.block_size

    def append_token(self, seq_id: int) -> int:
        """Reserve the slot for the sequence's next token and return it.

        A new block is taken when the last block is full; a shared last block
        (refcount > 1) is first copied to a new block (copy-on-write), and the
        (src, dst) pair is queued in ``self.copies``."""
        table = self.tables[seq_id]
        position = self.lengths[seq_id]
        logical = position // self.block_size
        if logical == len(table):
            table.append(self._allocate())
        else:
            block = table[logical]
            if self.refcount[block] > 1:
                fresh = self._allocate()
                self.copies.append((block, fresh))
                self.refcount[block] -= 1
                table[logical] = fresh
        self.lengths[seq_id] = position + 1
        return table[logical] * self.block_size + position % self.block_size

    def free_sequence(self, seq_id: int) -> None:
        """Drop a sequence; blocks whose count reaches zero return to the pool."""
        for block in self.tables.pop(seq_id):
            self._release(block)
        del self.lengths[seq_id]

    def take_copies(self) -> List[Tuple[int, int]]:
        """The copy-on-write pairs queued since the last call."""
        out, self.copies = self.copies, []
        return out

    # -- views --------------------------------------------------------------
    def table(self, seq_id: int) -> List[int]:
        return list(self.tables[seq_id])

    def length(self, seq_id: int) -> int:
        return self.lengths[seq_id]

    def num_free(self) -> int:
        return len(self.free)
