"""Named synthetic decode workloads.

Each preset describes the shape of one decode workload: dtype, head layout,
block size, how context lengths are drawn, how the physical pool is sized and
how many decode steps run.  The five presets follow the workloads that the
PagedAttention summary pages motivate (PagedAttention: Efficient LLM Serving
with vLLM, "The PagedAttention Algorithm" and "Advanced Features"):

  tiny_f32            4 sequences, 4 heads (MHA), head_dim 64, block 16,
                      lengths U{1..100}, a 64-block pool placed by a seeded
                      permutation, one decode step.
  llama7b_f16         Llama-7B-shaped decode: 32 heads = 32 kv heads, head_dim
                      128, block 16, batch 64, lengths U{128..2048}, pool 1.25x
                      the blocks needed, 100 decode steps.
  llama13b_cb_bf16    Llama-13B-shaped continuous batching: 40 heads, head_dim
                      128, block 16, batch 256, lengths lognormal (median 600,
                      sigma 0.8) clipped to [16, 4096]; each step 2% of the
                      sequences finish and are replaced by new ones of length
                      U{16..512} whose blocks come from a shuffled free list.
  shared_prefix_bf16  Parallel sampling: 32 prompts of length U{256..1024}, each
                      forked into 6 samples that alias the prompt's blocks;
                      GQA 32 q / 8 kv heads; 128 steps; copy-on-write of the
                      partially filled last prompt block at the first write.
  long_context_bf16   Long-context GQA decode: batch 16, 64 q / 8 kv heads,
                      lengths U{16384..32768}, block size 8/16/32, blocks
                      scattered over a ~60 GB pool, split-context partitions of
                      512 tokens.
  system_prompt_bf16  Prefix caching: 256 requests, each one of 4 system
                      prompts of U{1024..2048} tokens (request i takes prompt
                      i % 4, so sharers are spread through the batch) followed
                      by U{32..256} tokens of its own; the prompts' full blocks
                      are held once (a prefix cache's state), GQA 32 q / 8 kv
                      heads, 64 steps.

This module holds sizes only; the random draws live in ``workloads.gen``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

DTYPE_BYTES = {"f32": 4, "f16": 2, "bf16": 2}


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    dtype: str              # element type of q, k, v ("f32" | "f16" | "bf16")
    num_seqs: int           # batch of running sequences (B)
    num_heads: int          # query heads (H)
    num_kv_heads: int       # key/value heads (Hk); H / Hk query heads share one
    head_dim: int           # D
    block_size: int         # tokens per physical block (bs)
    steps: int              # decode steps of the workload
    lengths: str            # "uniform" | "lognormal"
    len_lo: int             # lower bound of the initial cached length
    len_hi: int             # upper bound of the initial cached length
    pool: str               # "fixed" | "factor" | "bytes"
    pool_value: float       # blocks, factor over need, or bytes
    kind: str = "plain"     # "plain" | "continuous" | "shared_prefix" | "system_prompt"
    lognormal_median: float = 600.0
    lognormal_sigma: float = 0.8
    replace_fraction: float = 0.0   # continuous batching: share finishing per step
    new_len_lo: int = 0
    new_len_hi: int = 0
    num_prompts: int = 0            # shared prefix: prompts, each forked
    samples_per_prompt: int = 0
    partition_size: int = 0         # 0 = let the library choose
    scale: float = 0.0              # 0 = 1/sqrt(head_dim)

    @property
    def elem_bytes(self) -> int:
        return DTYPE_BYTES[self.dtype]

    @property
    def group(self) -> int:
        return self.num_heads // self.num_kv_heads

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale > 0 else 1.0 / math.sqrt(self.head_dim)

    @property
    def kv_bytes_per_token(self) -> int:
        """Bytes of K plus V that one cached token holds in one layer."""
        return 2 * self.num_kv_heads * self.head_dim * self.elem_bytes

    @property
    def block_bytes(self) -> int:
        """Bytes of one physical block of ONE cache (K or V): [Hk, bs, D]."""
        return self.num_kv_heads * self.block_size * self.head_dim * self.elem_bytes

    def with_(self, **kw) -> "DecodeConfig":
        return replace(self, **kw)


TINY_F32 = DecodeConfig(
    name="tiny_f32", dtype="f32", num_seqs=4, num_heads=4, num_kv_heads=4,
    head_dim=64, block_size=16, steps=1, lengths="uniform", len_lo=1, len_hi=100,
    pool="fixed", pool_value=64, scale=1.0 / 8.0)

LLAMA7B_F16 = DecodeConfig(
    name="llama7b_f16", dtype="f16", num_seqs=64, num_heads=32, num_kv_heads=32,
    head_dim=128, block_size=16, steps=100, lengths="uniform", len_lo=128,
    len_hi=2048, pool="factor", pool_value=1.25)

LLAMA13B_CB_BF16 = DecodeConfig(
    name="llama13b_cb_bf16", dtype="bf16", num_seqs=256, num_heads=40,
    num_kv_heads=40, head_dim=128, block_size=16, steps=100, lengths="lognormal",
    len_lo=16, len_hi=4096, pool="factor", pool_value=1.5, kind="continuous",
    replace_fraction=0.02, new_len_lo=16, new_len_hi=512)

SHARED_PREFIX_BF16 = DecodeConfig(
    name="shared_prefix_bf16", dtype="bf16", num_seqs=192, num_heads=32,
    num_kv_heads=8, head_dim=128, block_size=16, steps=128, lengths="uniform",
    len_lo=256, len_hi=1024, pool="factor", pool_value=1.25, kind="shared_prefix",
    num_prompts=32, samples_per_prompt=6)

LONG_CONTEXT_BF16 = DecodeConfig(
    name="long_context_bf16", dtype="bf16", num_seqs=16, num_heads=64,
    num_kv_heads=8, head_dim=128, block_size=16, steps=10, lengths="uniform",
    len_lo=16384, len_hi=32768, pool="bytes", pool_value=60e9, partition_size=512)

SYSTEM_PROMPT_BF16 = DecodeConfig(
    name="system_prompt_bf16", dtype="bf16", num_seqs=256, num_heads=32, num_kv_heads=8,
    head_dim=128, block_size=16, steps=64, lengths="uniform", len_lo=1024, len_hi=2048,
    pool="factor", pool_value=1.25, kind="system_prompt", num_prompts=4, new_len_lo=32,
    new_len_hi=256)

CONFIGS = [TINY_F32, LLAMA7B_F16, LLAMA13B_CB_BF16, SHARED_PREFIX_BF16, LONG_CONTEXT_BF16,
           SYSTEM_PROMPT_BF16]
BY_NAME = {c.name: c for c in CONFIGS}
LONG_CONTEXT_BLOCK_SIZES = (8, 16, 32)


def get(name_or_index) -> DecodeConfig:
    if isinstance(name_or_index, int):
        return CONFIGS[name_or_index]
    if name_or_index.isdigit():
        return CONFIGS[int(name_or_index)]
    return BY_NAME[name_or_index]
