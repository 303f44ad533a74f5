"""The product's DecodeBatch / BlockPool and the oracle's prefix-cache model
driven through the same requests side by side.

Every call checks that the pool hands out what the oracle model does (tables,
cached-token counts, slots, copy pairs), so whatever tables and slots the
product produces here have been checked against the oracle before a kernel
sees them.  Scenarios follow the page "PagedAttention: Efficient LLM Serving
with vLLM", "Advanced Features": requests that share a system prompt (Prefix
Caching) and samples forked from one prompt (KV-Cache Sharing).
"""
from __future__ import annotations

import numpy as np

import paged_kv_cache_311_gb300 as pkv
from oracle.block_manager import OraclePrefixCache
from paged_kv_cache_311_gb300.batch import DecodeBatch


class Lockstep:
    def __init__(self, num_blocks: int, block_size: int, max_seqs: int, max_blocks_per_seq: int):
        self.bs = block_size
        self.pool = pkv.BlockPool(num_blocks, block_size)
        self.batch = DecodeBatch(self.pool, max_seqs, max_blocks_per_seq)
        self.model = OraclePrefixCache(num_blocks, block_size)
        self.mtab = {}
        self.mlen = {}

    def add(self, row: int, tokens, commit: bool = True):
        """A new request in `row`: -> (slots of its uncached tokens, cached tokens)."""
        tokens = np.asarray(tokens, dtype=np.int32)
        slots, cached = self.batch.add_prompt(row, tokens)
        want = self.model.allocate_prompt(tokens.tolist())
        assert want is not None
        n = -(-tokens.size // self.bs)
        assert self.batch.tables[row, :n].tolist() == want[0] and cached == want[1]
        self.mtab[row], self.mlen[row] = list(want[0]), int(tokens.size)
        pos = np.arange(cached, tokens.size)
        assert slots.tolist() == [want[0][p // self.bs] * self.bs + p % self.bs for p in pos]
        if commit:
            self.batch.commit(row, tokens)
            self.model.commit_prompt(tokens.tolist(), want[0])
        return slots, cached

    def fork(self, src: int, row: int) -> None:
        self.batch.fork(src, row)
        self.model.fork(self.mtab[src])
        self.mtab[row], self.mlen[row] = list(self.mtab[src]), self.mlen[src]

    def step(self, n: int):
        """One token more for rows 0..n-1: -> (slots, copy pairs), checked
        against the oracle model taking the rows one at a time in order."""
        slots, pairs = self.batch.step(n)
        want_pairs = []
        for row in range(n):
            slot, pair = self.model.append_token(self.mtab[row], self.mlen[row])
            self.mlen[row] += 1
            assert slots[row] == slot, (row, slots[row], slot)
            if pair:
                want_pairs.append(pair)
            L = self.mlen[row]
            assert self.batch.tables[row, : -(-L // self.bs)].tolist() == self.mtab[row]
            assert self.batch.lens[row] == L
        assert [tuple(p) for p in pairs.tolist()] == want_pairs
        return slots, pairs

    def check_holders(self) -> None:
        for b in range(self.model.num_blocks):
            assert self.pool.refcount(b) == self.model.holders[b]
            assert self.pool.is_cached(b) == self.model.is_cached(b)
        assert self.pool.available() == self.model.available()


def system_prompt_requests(seed: int, num_requests: int, num_prompts: int, prompt_lens, own_lens):
    """Request i: system prompt i % num_prompts followed by tokens of its own
    (token ids are arbitrary: only equality matters to the cache).
    -> (requests, prompts)."""
    rng = np.random.default_rng(seed)
    lo, hi = prompt_lens
    prompts = [rng.integers(0, 32000, int(rng.integers(lo, hi + 1))) for _ in range(num_prompts)]
    reqs = []
    for i in range(num_requests):
        own = rng.integers(0, 32000, int(rng.integers(own_lens[0], own_lens[1] + 1)))
        reqs.append(np.concatenate([prompts[i % num_prompts], own]).astype(np.int32))
    return reqs, prompts


def sampling_prompts(seed: int, num_prompts: int, prompt_lens):
    rng = np.random.default_rng(seed)
    lo, hi = prompt_lens
    return [rng.integers(0, 32000, int(rng.integers(lo, hi + 1))).astype(np.int32)
            for _ in range(num_prompts)]


def build_system_prompt(ls: Lockstep, reqs):
    """Every request in order (each committed at once): -> per-request
    (slots, cached tokens) of the prefill writes."""
    return [ls.add(i, r) for i, r in enumerate(reqs)]


def build_sampling(ls: Lockstep, prompts, samples: int):
    """Each prompt in rows p * samples, forked into the next samples - 1
    rows: -> per-prompt prefill (slots, cached tokens)."""
    pre = []
    for p, toks in enumerate(prompts):
        pre.append(ls.add(p * samples, toks, commit=False))
        for k in range(1, samples):
            ls.fork(p * samples, p * samples + k)
    return pre
