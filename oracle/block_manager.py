"""Reference KV block manager -- TEST INFRASTRUCTURE ONLY (see oracle/__init__).

Plain Python bookkeeping of physical blocks, written from the pages:

* a sequence of n tokens holds exactly ceil(n / block_size) blocks, taken on
  demand when a token starts a new block (PagedAttention: Efficient LLM
  Serving with vLLM, "The PagedAttention Algorithm", Steps 1-3, and "Memory
  Efficiency": 100 tokens at 16 per block -> 7 blocks, 112 slots, 12 unused);
* a page table maps logical block j to a physical block that may sit anywhere
  (same page, Step 4);
* sequences that share a prefix share its blocks; a shared block is copied on
  its first write, the way a forked process shares memory pages (same page, "Advanced Features", KV-Cache
  Sharing (Copy-on-Write)).

The refcount rule for the copy: a write into a block whose refcount is above
one allocates a fresh block, records (src, dst), drops the source's refcount
and points the writer's page table at the copy; a write into a block with
refcount one goes in place.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Tuple


def blocks_for_tokens(n_tokens: int, block_size: int) -> int:
    return -(-n_tokens // block_size)


class OracleBlockManager:
    def __init__(self, num_blocks: int, block_size: int, free_order: Optional[List[int]] = None):
        self.block_size = block_size
        self.num_blocks = num_blocks
        # Blocks are handed out from the end of this list.
        self.free: List[int] = list(free_order) if free_order is not None else list(range(num_blocks))[::-1]
        self.refcount = [0] * num_blocks
        self.tables: Dict[int, List[int]] = {}
        self.lengths: Dict[int, int] = {}

    # -- allocation -------------------------------------------------------
    def _take(self) -> int:
        if not self.free:
            raise MemoryError("no free block")
        b = self.free.pop()
        assert self.refcount[b] == 0
        self.refcount[b] = 1
        return b

    def add_sequence(self, seq: int, n_tokens: int) -> List[int]:
        table = [self._take() for _ in range(blocks_for_tokens(n_tokens, self.block_size))]
        self.tables[seq] = table
        self.lengths[seq] = n_tokens
        return list(table)

    def append_token(self, seq: int) -> Tuple[int, Optional[Tuple[int, int]]]:
        """Room for one more token: returns (slot, copy pair or None)."""
        table = self.tables[seq]
        pos = self.lengths[seq]
        j, off = divmod(pos, self.block_size)
        pair = None
        if off == 0:
            table.append(self._take())
        else:
            b = table[j]
            if self.refcount[b] > 1:
                nb = self._take()
                self.refcount[b] -= 1
                table[j] = nb
                pair = (b, nb)
        self.lengths[seq] = pos + 1
        return table[j] * self.block_size + off, pair

    def fork(self, parent: int, child: int) -> None:
        self.tables[child] = list(self.tables[parent])
        self.lengths[child] = self.lengths[parent]
        for b in self.tables[child]:
            self.refcount[b] += 1

    def free_sequence(self, seq: int) -> None:
        for b in self.tables.pop(seq):
            self.refcount[b] -= 1
            if self.refcount[b] == 0:
                self.free.append(b)
        self.lengths.pop(seq)

    # -- accounting -------------------------------------------------------
    def allocated_slots(self, seq: int) -> int:
        return len(self.tables[seq]) * self.block_size

    def unused_slots(self, seq: int) -> int:
        return self.allocated_slots(seq) - self.lengths[seq]
