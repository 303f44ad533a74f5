"""Moves a workload onto the GPU and runs its decode steps through the library.

Used by the GPU tests and the benchmark.  It holds no arithmetic of the
method: it allocates the caches with torch, fills them with the generator's
values, copies each step's inputs to the device and calls the library's three
operations in the order one decode step needs them (copy-on-write copies,
then the scatter of the new tokens, then attention).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

from .configs import DecodeConfig
from .gen import (TAG_CACHE_K, TAG_CACHE_V, TORCH_DTYPES, PagedDecodeWorkload, StepInputs,
                  fill_cache, step_values)


@dataclass
class DeviceStep:
    """One step's inputs resident on the device."""
    step: int
    q: torch.Tensor
    key: torch.Tensor
    value: torch.Tensor
    slot_mapping: torch.Tensor
    block_tables: torch.Tensor
    context_lens: torch.Tensor
    cow_pairs: Optional[torch.Tensor]
    max_context_len: int
    host: StepInputs
    plan: object = None                     # SharedPrefixPlan (shared-prefix workloads)
    plan_device: Optional[torch.Tensor] = None
    plan_seconds: float = 0.0               # host time the planner took for this step


class DeviceState:
    def __init__(self, cfg: DecodeConfig, workload: PagedDecodeWorkload, seed: int,
                 device="cuda", fill: bool = True, out_dtype: torch.dtype = torch.float32):
        self.cfg = cfg
        self.w = workload
        self.seed = seed
        self.device = torch.device(device)
        dt = TORCH_DTYPES[cfg.dtype]
        shape = (workload.num_blocks, cfg.num_kv_heads, cfg.block_size, cfg.head_dim)
        self.k_cache = torch.empty(shape, dtype=dt, device=self.device)
        self.v_cache = torch.empty(shape, dtype=dt, device=self.device)
        if fill:
            used = workload.used_blocks()
            fill_cache(self.k_cache, used, cfg.dtype, seed, TAG_CACHE_K)
            fill_cache(self.v_cache, used, cfg.dtype, seed, TAG_CACHE_V)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.out = torch.empty((workload.num_seqs, cfg.num_heads, cfg.head_dim), dtype=out_dtype,
                               device=self.device)
        self.workspace: Optional[torch.Tensor] = None

    def to_device(self, inp: StepInputs, value_device=None, shared: Optional[bool] = None,
                  partition_size: int = 0) -> DeviceStep:
        cfg, dev = self.cfg, self.device
        if shared is None:
            shared = cfg.kind in ("shared_prefix", "system_prompt")
        q, k, v = step_values(cfg, self.seed, inp, self.w.num_seqs,
                              device=value_device if value_device is not None else dev)
        pairs = None
        if inp.cow_pairs.shape[0]:
            pairs = torch.as_tensor(inp.cow_pairs, dtype=torch.int64).to(dev)
        plan = plan_dev = None
        plan_s = 0.0
        if shared:
            import time

            import paged_kv_cache_311_gb300 as pkv
            t0 = time.perf_counter()
            plan = pkv.plan_shared_prefix(inp.block_tables, inp.context_lens, cfg.num_heads,
                                          cfg.num_kv_heads, cfg.head_dim, cfg.block_size,
                                          inp.max_context_len, partition_size)
            plan_s = time.perf_counter() - t0
            plan_dev = plan.to(dev)
        return DeviceStep(
            step=inp.step, q=q.to(dev), key=k.to(dev), value=v.to(dev),
            slot_mapping=torch.as_tensor(inp.slot_mapping).to(dev),
            block_tables=torch.as_tensor(inp.block_tables).to(dev),
            context_lens=torch.as_tensor(inp.context_lens).to(dev),
            cow_pairs=pairs, max_context_len=inp.max_context_len, host=inp,
            plan=plan, plan_device=plan_dev, plan_seconds=plan_s)

    def ensure_workspace(self, max_context_len: int, partition_size: int,
                         plan=None) -> None:
        import paged_kv_cache_311_gb300 as pkv
        if plan is not None:
            need = plan.workspace_bytes
        else:
            need = pkv.paged_attention_workspace_bytes(self.w.num_seqs, self.cfg.num_heads,
                                                       max_context_len, self.cfg.head_dim,
                                                       partition_size)
        if need and (self.workspace is None or self.workspace.numel() < need):
            self.workspace = torch.empty(need, dtype=torch.uint8, device=self.device)

    def run_step(self, s: DeviceStep, partition_size: Optional[int] = None,
                 out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        """copy_blocks (if the step has copy-on-write pairs), reshape_and_cache,
        then paged attention -- all on the current stream.  A step that
        carries a shared-prefix plan takes the shared-prefix entry point."""
        import paged_kv_cache_311_gb300 as pkv
        cfg = self.cfg
        P = cfg.partition_size if partition_size is None else partition_size
        out = self.out if out is None else out
        if s.cow_pairs is not None:
            pkv.copy_blocks([self.k_cache], [self.v_cache], s.cow_pairs,
                            device_status=self.status, stream=stream)
        pkv.reshape_and_cache(s.key, s.value, self.k_cache, self.v_cache, s.slot_mapping,
                              device_status=self.status, stream=stream)
        self.ensure_workspace(s.max_context_len, P, s.plan)
        if s.plan is not None:
            pkv.paged_attention_decode_shared(
                out, s.q, self.k_cache, self.v_cache, s.block_tables, s.context_lens,
                cfg.softmax_scale, s.plan, s.plan_device, max_context_len=s.max_context_len,
                workspace=self.workspace, device_status=self.status, stream=stream)
        else:
            pkv.paged_attention_decode(
                out, s.q, self.k_cache, self.v_cache, s.block_tables, s.context_lens,
                cfg.softmax_scale, max_context_len=s.max_context_len, partition_size=P,
                workspace=self.workspace, device_status=self.status, stream=stream)
        return out


def algorithmic_bytes(cfg: DecodeConfig, inp: StepInputs, num_seqs: int, split_partition: int = 0,
                      out_bytes: int = 4, partials=None) -> dict:
    """Bytes one decode step must move at minimum.

    attention: every distinct (physical block, kv head, row) slot that some
    sequence reads (logical position < its context length), K and V, once;
    plus q, the output, the block-table entries and context lengths; plus the
    split path's workspace round trip when it runs (one partial per head and
    non-empty partition of split_partition tokens, or `partials[s]` per head
    of sequence s for a shared-prefix plan; none when partials[s] is 1, since
    the one item that holds such a sequence writes its output directly).
    Shared prefix blocks count once.  scatter: the new tokens' K/V read once and written once.
    copy: each copied block read once and written once."""
    bs, e = cfg.block_size, cfg.elem_bytes
    row = cfg.head_dim * e
    slots = set()
    logical = 0
    table_entries = 0
    for s in range(num_seqs):
        L = int(inp.context_lens[s])
        nb = -(-L // bs)
        table_entries += nb
        logical += L
        tb = inp.block_tables[s]
        for j in range(nb):
            rows = min(bs, L - j * bs)
            slots.add((int(tb[j]), rows))
    # distinct rows: a block shared by several sequences is read up to the
    # longest prefix any of them covers
    per_block = {}
    for b, rows in slots:
        per_block[b] = max(per_block.get(b, 0), rows)
    distinct_rows = sum(per_block.values())
    kv = 2 * distinct_rows * cfg.num_kv_heads * row
    qo = num_seqs * cfg.num_heads * cfg.head_dim * (e + out_bytes)
    meta = table_entries * 4 + num_seqs * 4
    ws = 0
    if split_partition:
        parts = sum(-(-int(L) // split_partition) for L in inp.context_lens[:num_seqs])
        ws = 2 * cfg.num_heads * parts * (cfg.head_dim + 2) * 4
    if partials is not None:
        merged = np.asarray(partials)
        ws = 2 * cfg.num_heads * int(np.sum(merged[merged > 1])) * (cfg.head_dim + 2) * 4
    attn = kv + qo + meta + ws
    T = inp.num_tokens
    scatter = 2 * 2 * T * cfg.num_kv_heads * row + T * 8
    copy = 2 * 2 * inp.cow_pairs.shape[0] * cfg.block_bytes
    return dict(attention=attn, kv=kv, logical_kv=2 * logical * cfg.num_kv_heads * row,
                scatter=scatter, copy=copy, total=attn + scatter + copy)
