"""Host-side block bookkeeping for building block tables, slot mappings and
copy-on-write pairs.

This is the allocator side of paged KV caching as the pages describe it: a
pool of fixed-size physical blocks, a per-request block table mapping logical
block j to a physical block ("vLLM intro part 2", section 3.2), reference
counts on shared blocks, and the copy-on-write rule -- before writing into a
block whose reference count is above one, take a fresh block, copy the old
block into it, point the request's table at it, drop one reference from the
old block and then write ("vLLM intro part 2", section 5; aibook
"显存与 KV 缓存", the five copy-on-write steps and the ``append_kv`` fix that
checks the block's own count).

It produces the integer inputs of the GPU path (tables, slots, copy pairs);
it does no attention arithmetic.  Free blocks are handed out in the order
given at construction (tests pass a seeded random permutation, so physical
placement is arbitrary, as the pages stress).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple


@dataclass
class SeqState:
    table: List[int] = field(default_factory=list)
    length: int = 0


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int, order: Optional[Sequence[int]] = None):
        if block_size <= 0 or num_blocks <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = num_blocks
        self.block_size = block_size
        order = list(range(num_blocks)) if order is None else [int(b) for b in order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("order must be a permutation of the block ids")
        self._free = order[::-1]          # pop() from the end hands out order[0] first
        self.ref_cnt = [0] * num_blocks
        self.seqs: List[SeqState] = []
        self.cow_pairs: List[Tuple[int, int]] = []

    # -- blocks -------------------------------------------------------------
    def num_free(self) -> int:
        return len(self._free)

    def allocate(self) -> int:
        if not self._free:
            raise MemoryError("block pool exhausted")
        b = self._free.pop()
        self.ref_cnt[b] = 1
        return b

    def _release(self, b: int) -> None:
        if self.ref_cnt[b] <= 0:
            raise RuntimeError(f"block {b} released with ref_cnt {self.ref_cnt[b]}")
        self.ref_cnt[b] -= 1
        if self.ref_cnt[b] == 0:
            self._free.append(b)

    # -- sequences ----------------------------------------------------------
    def new_sequence(self) -> int:
        self.seqs.append(SeqState())
        return len(self.seqs) - 1

    def fork(self, parent: int) -> int:
        """A new sequence sharing every block of ``parent`` (ref_cnt += 1)."""
        src = self.seqs[parent]
        child = SeqState(table=list(src.table), length=src.length)
        for b in child.table:
            self.ref_cnt[b] += 1
        self.seqs.append(child)
        return len(self.seqs) - 1

    def append_slot(self, seq: int) -> int:
        """Reserve the slot for the next token of ``seq`` and return it.

        A position at a block boundary takes a fresh block.  A position inside
        a block shared with other sequences triggers copy-on-write: the pair
        (old, new) is recorded in ``cow_pairs`` and the table repointed before
        the slot is returned, so the caller copies first and writes after.
        """
        s = self.seqs[seq]
        pos = s.length
        j, off = divmod(pos, self.block_size)
        if off == 0:
            s.table.append(self.allocate())
        else:
            old = s.table[j]
            if self.ref_cnt[old] > 1:
                new = self.allocate()
                self.cow_pairs.append((old, new))
                s.table[j] = new
                self.ref_cnt[old] -= 1
        s.length = pos + 1
        return s.table[j] * self.block_size + off

    def free_sequence(self, seq: int) -> None:
        """Drop the sequence's references, last block first."""
        s = self.seqs[seq]
        for b in reversed(s.table):
            self._release(b)
        s.table = []
        s.length = 0

    def take_cow_pairs(self) -> List[Tuple[int, int]]:
        pairs, self.cow_pairs = self.cow_pairs, []
        return pairs
