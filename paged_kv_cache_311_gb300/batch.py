"""Host bookkeeping of a decode batch over one BlockPool.

The block pool's calls in the order a serving loop makes them for one paged
cache (PagedAttention: Efficient LLM Serving with vLLM, "The PagedAttention
Algorithm", Steps 1-3, and "Advanced Features", KV-Cache Sharing and Prefix
Caching):

* a new request's prompt gets its blocks (``add_prompt``): the full blocks the
  prefix cache holds for exactly its leading tokens are reused, fresh blocks
  take the rest, and the slots of the tokens the cache did not hold come back
  for the prefill's ``reshape_and_cache``; once that K/V is written the prompt
  is committed (``commit``), so later requests reuse its full blocks;
* a forked sample holds every block of its parent (``fork``);
* each decode step gives every running sequence the slot of its next token in
  one ``append_slots`` call (``step``): a fresh block when the token starts
  one, a copy first when the last block is shared or cached; the copy pairs
  go to ``copy_blocks``;
* a finished sequence lets go of its blocks (``release``).

Rows of ``tables`` / ``lens`` are the batch's sequences; the kernels take
``tables[:n]`` and ``lens[:n]`` as block_tables and context_lens.  Nothing
here computes attention.
"""
from __future__ import annotations

from typing import Optional, Tuple

import numpy as np


class DecodeBatch:
    def __init__(self, pool, max_seqs: int, max_blocks_per_seq: int):
        self.pool = pool
        self.block_size = pool.block_size
        self.tables = np.full((max_seqs, max_blocks_per_seq), -1, np.int32)
        self.lens = np.zeros(max_seqs, np.int32)
        self.live = np.zeros(max_seqs, bool)

    def _blocks(self, row: int) -> np.ndarray:
        return self.tables[row, : -(-int(self.lens[row]) // self.block_size)]

    def add_prompt(self, row: int, tokens) -> Tuple[np.ndarray, int]:
        """Row `row` (free) becomes a request holding `tokens`: -> (slots of
        the tokens the prefix cache did not hold, int64; cached tokens)."""
        assert not self.live[row]
        tokens = np.asarray(tokens)
        n, bs = int(tokens.size), self.block_size
        table, cached = self.pool.allocate_prompt(tokens)
        if table.size > self.tables.shape[1]:
            self.pool.release(table)
            raise ValueError("prompt longer than the table rows")
        self.tables[row, :] = -1
        self.tables[row, : table.size] = table
        self.lens[row] = n
        self.live[row] = True
        pos = np.arange(cached, n, dtype=np.int64)
        return table[pos // bs].astype(np.int64) * bs + pos % bs, cached

    def commit(self, row: int, tokens) -> None:
        """The K/V of row's prompt is written: cache its full blocks."""
        self.pool.commit_prompt(np.asarray(tokens), self._blocks(row))

    def fork(self, src: int, row: int) -> None:
        """Row `row` (free) becomes a sample of `src`, holding its blocks."""
        assert self.live[src] and not self.live[row]
        self.pool.fork(self._blocks(src))
        self.tables[row] = self.tables[src]
        self.lens[row] = self.lens[src]
        self.live[row] = True

    def release(self, row: int) -> None:
        self.pool.release(self._blocks(row))
        self.tables[row, :] = -1
        self.lens[row] = 0
        self.live[row] = False

    def step(self, n: Optional[int] = None) -> Tuple[np.ndarray, np.ndarray]:
        """One more token for each of rows 0..n-1 (all live), in batch order:
        -> (slots int64 [n], copy pairs int64 [k, 2]); lens grow by one."""
        n = int(self.live.sum()) if n is None else n
        assert self.live[:n].all()
        slots, pairs = self.pool.append_slots(self.tables[:n], self.lens[:n])
        self.lens[:n] += 1
        return slots, pairs
