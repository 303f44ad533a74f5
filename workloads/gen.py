"""Seeded input generator for paged decode workloads.

What this module draws, and nothing more:
  * context lengths (uniform or clipped lognormal),
  * where each sequence's blocks sit in the physical pool (a seeded permutation
    of the pool, or pops from uniformly random positions of the free list for
    the continuous-batching preset),
  * per decode step: which slot each new token goes to, the block tables, the
    context lengths, and the (source, destination) block pairs that a
    copy-on-write of a shared block needs,
  * the N(0,1) values of q, the new tokens' k and v, and the initial cache
    contents, rounded to the workload dtype.

It computes no attention, no cache scatter and no block copy: the CUDA library
and the CPU oracle both take its output as input.  Structure draws use numpy's
Philox generator; value draws use torch's generator on the requested device.

Blocks are handed out on demand: a sequence whose next token starts a new
block position (length % block_size == 0) takes one block from the free list
(PagedAttention: Efficient LLM Serving with vLLM, "The PagedAttention
Algorithm", Steps 1-3).  Shared-prefix samples alias the prompt's blocks and a
block shared by more than one sequence is copied before its first write
("Advanced Features", KV-Cache Sharing (Copy-on-Write)).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch

from .configs import DecodeConfig

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass
class StepInputs:
    """Everything one decode step hands to the kernels (host arrays)."""
    step: int
    slot_mapping: np.ndarray        # int64 [T]; token t goes to slot slot_mapping[t]
    token_seq: np.ndarray           # int64 [T]; sequence that owns token t
    token_pos: np.ndarray           # int64 [T]; logical position of token t
    context_lens: np.ndarray        # int32 [B]; tokens attended, incl. this step's
    block_tables: np.ndarray        # int32 [B, MB]; unused entries are -1
    cow_pairs: np.ndarray           # int64 [P, 2]; (src, dst) block copies before the scatter
    max_context_len: int

    @property
    def num_tokens(self) -> int:
        return int(self.slot_mapping.shape[0])


class _FreeList:
    """Pool of free physical block ids.

    ``pop`` takes either the last entry (drawing from a seeded permutation) or
    the entry at a uniformly random position (a shuffled free list)."""

    def __init__(self, order: np.ndarray, rng: np.random.Generator, random_pop: bool):
        self.ids = np.array(order, dtype=np.int64)
        self.count = int(self.ids.shape[0])
        self.rng = rng
        self.random_pop = random_pop

    def pop(self) -> int:
        if self.count == 0:
            raise RuntimeError("physical block pool exhausted")
        if self.random_pop:
            i = int(self.rng.integers(0, self.count))
        else:
            i = self.count - 1
        b = int(self.ids[i])
        self.ids[i] = self.ids[self.count - 1]
        self.count -= 1
        return b

    def push(self, b: int) -> None:
        if self.count == self.ids.shape[0]:
            self.ids = np.concatenate([self.ids, np.zeros_like(self.ids)])
        self.ids[self.count] = b
        self.count += 1


def _blocks_for(n_tokens: int, bs: int) -> int:
    return -(-n_tokens // bs)


@dataclass
class _Seq:
    table: List[int] = field(default_factory=list)
    length: int = 0                 # tokens already in the cache


class PagedDecodeWorkload:
    """Host-side simulation of a batch of decoding sequences over a block pool.

    ``setup`` state: every running sequence holds its initial tokens (their
    k/v are the initial cache contents).  Each ``next_step`` appends exactly
    one decode token per running sequence (plus, for the continuous-batching
    preset, the prompt tokens of the sequences that replace finished ones).
    """

    def __init__(self, cfg: DecodeConfig, seed: int, *, pool_blocks: Optional[int] = None,
                 total_steps: Optional[int] = None, num_seqs: Optional[int] = None,
                 contiguous: bool = False):
        self.cfg = cfg
        self.seed = int(seed)
        self.rng = np.random.Generator(np.random.Philox(self.seed))
        self.bs = cfg.block_size
        self.total_steps = cfg.steps if total_steps is None else int(total_steps)
        B = cfg.num_seqs if num_seqs is None else int(num_seqs)
        self.step_index = 0
        self.refcount: Optional[np.ndarray] = None

        if cfg.kind == "shared_prefix":
            P = cfg.num_prompts if num_seqs is None else max(1, B // cfg.samples_per_prompt)
            self.prompt_lens = self.rng.integers(cfg.len_lo, cfg.len_hi + 1, size=P)
            init_lens = np.repeat(self.prompt_lens, cfg.samples_per_prompt)
            B = int(init_lens.shape[0])
        elif cfg.kind == "system_prompt":
            # request i starts with system prompt i % P, then its own tokens
            self.prompt_lens = self.rng.integers(cfg.len_lo, cfg.len_hi + 1, size=cfg.num_prompts)
            self.own_lens = self.rng.integers(cfg.new_len_lo, cfg.new_len_hi + 1, size=B)
            self.prompt_of = np.arange(B) % cfg.num_prompts
            init_lens = self.prompt_lens[self.prompt_of] + self.own_lens
        else:
            init_lens = self._draw_lengths(B, cfg.len_lo, cfg.len_hi)
        self.num_seqs = B
        self.init_lens = init_lens.astype(np.int64)

        # Longest context any sequence can reach over the run.
        longest_new = cfg.new_len_hi if cfg.kind == "continuous" else 0
        self.max_len_total = int(max(self.init_lens.max(), longest_new)) + self.total_steps
        self.max_blocks_per_seq = _blocks_for(self.max_len_total, self.bs)

        # Pool size.
        if pool_blocks is not None:
            nb = int(pool_blocks)
        elif cfg.pool == "fixed":
            nb = int(cfg.pool_value)
        elif cfg.pool == "factor":
            nb = int(math.ceil(cfg.pool_value * self._peak_blocks_needed()))
        elif cfg.pool == "bytes":
            nb = int(cfg.pool_value // (2 * cfg.block_bytes))
        else:
            raise ValueError(cfg.pool)
        self.num_blocks = nb
        order = self.rng.permutation(nb)
        pop_rng = np.random.Generator(np.random.Philox(_stream_seed(self.seed, 99)))
        self.free = _FreeList(order, pop_rng, random_pop=(cfg.kind == "continuous"))

        # Initial placement.
        self.seqs: List[_Seq] = []
        self.reserved_next: Optional[List[int]] = None
        if contiguous:
            # Every sequence owns one run of consecutive blocks big enough for
            # its whole run (the layout of a contiguous, non-paged cache).
            if cfg.kind != "plain":
                raise ValueError("contiguous placement is defined for plain workloads only")
            need = [_blocks_for(int(L) + self.total_steps, self.bs) for L in self.init_lens]
            if sum(need) > nb:
                raise ValueError("pool too small for contiguous placement")
            base = 0
            self.reserved_next = []
            for L, n in zip(self.init_lens, need):
                k = _blocks_for(int(L), self.bs)
                self.seqs.append(_Seq(table=list(range(base, base + k)), length=int(L)))
                self.reserved_next.append(base + k)
                base += n
            return
        if cfg.kind == "shared_prefix":
            self.refcount = np.zeros(nb, dtype=np.int32)
            S = cfg.samples_per_prompt
            for p, lp in enumerate(self.prompt_lens):
                table = [self.free.pop() for _ in range(_blocks_for(int(lp), self.bs))]
                for b in table:
                    self.refcount[b] = S
                for _ in range(S):
                    self.seqs.append(_Seq(table=list(table), length=int(lp)))
        elif cfg.kind == "system_prompt":
            # A prefix cache holds the full blocks of each system prompt once;
            # a request's own blocks hold the prompt's partial last block (if
            # any) and its own tokens.
            self.refcount = np.zeros(nb, dtype=np.int32)
            shared = [[self.free.pop() for _ in range(int(lp) // self.bs)] for lp in self.prompt_lens]
            for i, L in enumerate(self.init_lens):
                base = shared[self.prompt_of[i]]
                own = [self.free.pop() for _ in range(_blocks_for(int(L), self.bs) - len(base))]
                for b in base:
                    self.refcount[b] += 1
                for b in own:
                    self.refcount[b] = 1
                self.seqs.append(_Seq(table=list(base) + own, length=int(L)))
        else:
            for L in self.init_lens:
                table = [self.free.pop() for _ in range(_blocks_for(int(L), self.bs))]
                self.seqs.append(_Seq(table=table, length=int(L)))

    # ------------------------------------------------------------------ draws
    def _draw_lengths(self, n: int, lo: int, hi: int) -> np.ndarray:
        cfg = self.cfg
        if cfg.lengths == "uniform":
            return self.rng.integers(lo, hi + 1, size=n)
        if cfg.lengths == "lognormal":
            z = self.rng.standard_normal(n)
            L = np.rint(cfg.lognormal_median * np.exp(cfg.lognormal_sigma * z))
            return np.clip(L, lo, hi).astype(np.int64)
        raise ValueError(cfg.lengths)

    def _peak_blocks_needed(self) -> int:
        """Blocks in use at the busiest point of the run, found by a dry run of
        the same draws on a copy of the generator state."""
        cfg = self.cfg
        saved = self.rng.bit_generator.state
        try:
            if cfg.kind == "shared_prefix":
                S = cfg.samples_per_prompt
                total = 0
                for lp in self.prompt_lens:
                    shared = _blocks_for(int(lp), self.bs)
                    own = S * (_blocks_for(int(lp) + self.total_steps, self.bs) - (int(lp) // self.bs))
                    total += shared + own
                return total
            if cfg.kind == "system_prompt":
                shared = sum(int(lp) // self.bs for lp in self.prompt_lens)
                own = sum(_blocks_for(int(L) + self.total_steps, self.bs) -
                          int(self.prompt_lens[self.prompt_of[i]]) // self.bs
                          for i, L in enumerate(self.init_lens))
                return shared + own
            if cfg.kind == "continuous":
                lens = self.init_lens.copy()
                in_use = int(sum(_blocks_for(int(L), self.bs) for L in lens))
                peak = in_use
                n_rep = int(round(cfg.replace_fraction * self.num_seqs))
                for _ in range(self.total_steps):
                    if n_rep:
                        done = self.rng.choice(self.num_seqs, size=n_rep, replace=False)
                        new = self.rng.integers(cfg.new_len_lo, cfg.new_len_hi + 1, size=n_rep)
                        for s, L in zip(done, new):
                            in_use -= _blocks_for(int(lens[s]), self.bs)
                            lens[s] = int(L)
                            in_use += _blocks_for(int(L), self.bs)
                    grow = int(np.sum(lens % self.bs == 0))
                    lens += 1
                    in_use += grow
                    peak = max(peak, in_use)
                return peak
            return int(sum(_blocks_for(int(L) + self.total_steps, self.bs) for L in self.init_lens))
        finally:
            self.rng.bit_generator.state = saved

    # ------------------------------------------------------------ accessors
    def used_blocks(self) -> np.ndarray:
        """Physical blocks that hold cached tokens right now (sorted, unique)."""
        s = set()
        for q in self.seqs:
            s.update(q.table)
        return np.array(sorted(s), dtype=np.int64)

    def context_lens(self) -> np.ndarray:
        return np.array([q.length for q in self.seqs], dtype=np.int32)

    def block_tables(self) -> np.ndarray:
        t = np.full((self.num_seqs, self.max_blocks_per_seq), -1, dtype=np.int32)
        for i, q in enumerate(self.seqs):
            t[i, :len(q.table)] = q.table
        return t

    # ----------------------------------------------------------------- step
    def _append(self, s: int, cow: list) -> tuple:
        """Give sequence s one more token; returns (slot, position)."""
        q = self.seqs[s]
        pos = q.length
        j, o = divmod(pos, self.bs)
        if o == 0:
            if self.reserved_next is not None:
                b = self.reserved_next[s]
                self.reserved_next[s] += 1
            else:
                b = self.free.pop()
            q.table.append(b)
            if self.refcount is not None:
                self.refcount[b] = 1
        else:
            b = q.table[j]
            if self.refcount is not None and self.refcount[b] > 1:
                nb = self.free.pop()
                cow.append((b, nb))
                self.refcount[b] -= 1
                self.refcount[nb] = 1
                q.table[j] = nb
                b = nb
        q.length += 1
        return b * self.bs + o, pos

    def _release(self, s: int) -> None:
        q = self.seqs[s]
        for b in q.table:
            if self.refcount is not None:
                self.refcount[b] -= 1
                if self.refcount[b] > 0:
                    continue
            self.free.push(b)
        q.table = []
        q.length = 0

    def next_step(self) -> StepInputs:
        cfg = self.cfg
        slots, owners, positions, cow = [], [], [], []
        if cfg.kind == "continuous":
            n_rep = int(round(cfg.replace_fraction * self.num_seqs))
            if n_rep:
                done = self.rng.choice(self.num_seqs, size=n_rep, replace=False)
                new = self.rng.integers(cfg.new_len_lo, cfg.new_len_hi + 1, size=n_rep)
                for s, L in zip(done, new):
                    self._release(int(s))
                    for _ in range(int(L)):
                        sl, pos = self._append(int(s), cow)
                        slots.append(sl); owners.append(int(s)); positions.append(pos)
        for s in range(self.num_seqs):
            sl, pos = self._append(s, cow)
            slots.append(sl); owners.append(s); positions.append(pos)
        lens = self.context_lens()
        inp = StepInputs(
            step=self.step_index,
            slot_mapping=np.array(slots, dtype=np.int64),
            token_seq=np.array(owners, dtype=np.int64),
            token_pos=np.array(positions, dtype=np.int64),
            context_lens=lens,
            block_tables=self.block_tables(),
            cow_pairs=np.array(cow, dtype=np.int64).reshape(-1, 2),
            max_context_len=int(lens.max()) if lens.size else 0,
        )
        self.step_index += 1
        return inp


# ------------------------------------------------------------------ values
def _stream_seed(seed: int, *tags: int) -> int:
    """Derive an independent 63-bit seed for one value stream."""
    ss = np.random.SeedSequence([int(seed)] + [int(t) for t in tags])
    return int(ss.generate_state(1, dtype=np.uint64)[0] & ((1 << 63) - 1))


def normal(shape, dtype: str, seed: int, *tags: int, device="cpu") -> torch.Tensor:
    """N(0,1) values drawn in fp32 and rounded to ``dtype`` (round to nearest even)."""
    g = torch.Generator(device=device)
    g.manual_seed(_stream_seed(seed, *tags))
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32, device=device)
    return x.to(TORCH_DTYPES[dtype])


# Value-stream tags.
TAG_Q, TAG_K, TAG_V, TAG_CACHE_K, TAG_CACHE_V = 1, 2, 3, 4, 5


def step_values(cfg: DecodeConfig, seed: int, inp: StepInputs, num_seqs: int, device="cpu"):
    """q [B, H, D] and the new tokens' key/value [T, Hk, D] of one step."""
    q = normal((num_seqs, cfg.num_heads, cfg.head_dim), cfg.dtype, seed, TAG_Q, inp.step, device=device)
    k = normal((inp.num_tokens, cfg.num_kv_heads, cfg.head_dim), cfg.dtype, seed, TAG_K, inp.step, device=device)
    v = normal((inp.num_tokens, cfg.num_kv_heads, cfg.head_dim), cfg.dtype, seed, TAG_V, inp.step, device=device)
    return q, k, v


def fill_cache(cache: torch.Tensor, blocks: np.ndarray, dtype: str, seed: int, tag: int,
               chunk_blocks: int = 4096) -> None:
    """Write N(0,1) values into the given physical blocks of ``cache``
    ([NB, Hk, bs, D]); blocks are processed in fixed-size chunks so the
    values depend only on the seed and the block list."""
    per_block = tuple(cache.shape[1:])
    idx_all = torch.as_tensor(np.asarray(blocks, dtype=np.int64))
    for c, start in enumerate(range(0, idx_all.numel(), chunk_blocks)):
        idx = idx_all[start:start + chunk_blocks].to(cache.device)
        vals = normal((idx.numel(),) + per_block, dtype, seed, tag, c, device=cache.device)
        cache.index_copy_(0, idx, vals)
