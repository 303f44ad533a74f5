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


class OraclePrefixCache:
    """Block manager with prefix caching, for requests given as token ids.

    Written from the page "PagedAttention: Efficient LLM Serving with vLLM":

    * blocks are taken on demand and held by reference count; a write into a
      block that another sequence also holds goes to a copy first ("The
      PagedAttention Algorithm", Steps 1-3; "Advanced Features", KV-Cache
      Sharing: only the divergent tokens get new blocks);
    * "Advanced Features", Prefix Caching: the first request with a given
      prefix computes its KV blocks and they are cached; a later request
      that starts with the same tokens reuses them instead of computing them.

    Readings where the page is silent:

    * Only FULL blocks are cached, and a block is identified by every token
      from the start of the prompt to its own end: its K/V depend on all of
      them.  The key here is that whole token prefix itself (no hash), so a
      hit is exact by construction.  A request reuses the longest run of
      leading full blocks whose prefixes are cached.
    * A block enters the cache when the caller commits the prompt, after its
      K/V has been written.  A cached block is never written in place (every
      later reuser reads it): a write into it goes to a copy, even when the
      writer is its only holder.
    * A cached block that no sequence holds keeps its entry and stays
      reusable.  When a fresh block is needed and none is free, the cached
      block released longest ago is taken and its entry dropped.
    * A request that cannot get all its blocks takes nothing and changes
      nothing.
    * Free blocks are handed out last-freed first, block 0 first in a new
      pool, as OracleBlockManager does.
    """

    def __init__(self, num_blocks: int, block_size: int):
        self.block_size = block_size
        self.num_blocks = num_blocks
        self.free: List[int] = list(range(num_blocks))[::-1]
        self.holders = [0] * num_blocks
        self.entry: Dict[Tuple[int, ...], int] = {}    # token prefix -> block ending it
        self.key: Dict[int, Tuple[int, ...]] = {}      # cached block -> its prefix
        self.idle: List[int] = []    # cached blocks nobody holds, released longest ago first
        self.lookups = 0
        self.hits = 0

    def available(self) -> int:
        return len(self.free) + len(self.idle)

    def _prefix(self, toks: Tuple[int, ...], k: int) -> Tuple[int, ...]:
        """Cache key of logical block k: every token up to the block's end."""
        return toks[:(k + 1) * self.block_size]

    def is_cached(self, b: int) -> bool:
        return b in self.key

    def _take(self) -> int:
        if self.free:
            b = self.free.pop()
        else:
            b = self.idle.pop(0)           # released longest ago
            del self.entry[self.key.pop(b)]
        self.holders[b] = 1
        return b

    def _hold(self, b: int) -> None:
        if self.holders[b] == 0 and b in self.key:
            self.idle.remove(b)
        self.holders[b] += 1

    def _let_go(self, b: int) -> None:
        self.holders[b] -= 1
        if self.holders[b] == 0:
            if b in self.key:
                self.idle.append(b)
            else:
                self.free.append(b)

    def allocate_prompt(self, tokens) -> Optional[Tuple[List[int], int]]:
        """(table, cached tokens) for a new request, or None with nothing taken."""
        bs, toks = self.block_size, tuple(int(t) for t in tokens)
        reused: List[int] = []
        for k in range(len(toks) // bs):
            self.lookups += 1
            b = self.entry.get(self._prefix(toks, k))
            if b is None:
                break
            self.hits += 1
            reused.append(b)
        fresh = blocks_for_tokens(len(toks), bs) - len(reused)
        idle_reused = sum(1 for b in reused if self.holders[b] == 0)
        if self.available() - idle_reused < fresh:
            return None
        for b in reused:
            self._hold(b)
        return reused + [self._take() for _ in range(fresh)], len(reused) * bs

    def commit_prompt(self, tokens, table) -> None:
        """The prompt's K/V is written: its full blocks become cache entries
        (a prefix that already has an entry keeps it)."""
        bs, toks = self.block_size, tuple(int(t) for t in tokens)
        for k in range(len(toks) // bs):
            prefix, b = self._prefix(toks, k), int(table[k])
            if b not in self.key and prefix not in self.entry:
                self.entry[prefix] = b
                self.key[b] = prefix

    def allocate(self, n: int) -> Optional[List[int]]:
        if self.available() < n:
            return None
        return [self._take() for _ in range(n)]

    def fork(self, table) -> None:
        for b in table:
            self._hold(int(b))

    def release(self, table) -> None:
        for b in table:
            self._let_go(int(b))

    def prepare_write(self, table: List[int], j: int) -> Optional[Tuple[int, int]]:
        """Before a write into table[j]: the (old, copy) pair when the block
        is shared or cached (table[j] then names the copy), else None."""
        b = table[j]
        if self.holders[b] == 1 and b not in self.key:
            return None
        if self.available() < 1:
            raise MemoryError("no block for the copy")
        nb = self._take()
        self._let_go(b)
        table[j] = nb
        return b, nb

    def append_token(self, table: List[int], length: int) -> Tuple[int, Optional[Tuple[int, int]]]:
        """Room for token `length` of a sequence holding `length` tokens in
        `table` (updated in place): its slot, and the copy pair if any."""
        j, off = divmod(length, self.block_size)
        pair = None
        if off == 0:
            got = self.allocate(1)
            if got is None:
                raise MemoryError("no free block")
            table.append(got[0])
        else:
            pair = self.prepare_write(table, j)
        return table[j] * self.block_size + off, pair
