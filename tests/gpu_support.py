"""GPU-test helpers: run the library on a case and compute the oracle's answer.

The oracle never reads anything the CUDA path produced: its cache copies are
taken from the generator's values before any library kernel runs, and it
applies its own scatter and copy-on-write copies to them."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from tests.util import raw_np

TOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 2e-3}


def gpu_decode(case, partition_size=0, out_dtype=torch.float32, max_context_len=None,
               engine="auto"):
    import paged_kv_cache_311_gb300 as pkv
    pkv.set_decode_engine(engine)
    dev = torch.device("cuda")
    q = case["q"].to(dev)
    kc = case["k_cache"].to(dev)
    vc = case["v_cache"].to(dev)
    bt = torch.as_tensor(case["block_tables"], dtype=torch.int32).to(dev)
    cl = torch.as_tensor(case["context_lens"], dtype=torch.int32).to(dev)
    out = torch.full(q.shape, float("nan"), dtype=out_dtype, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    mcl = int(max(case["context_lens"])) if max_context_len is None else max_context_len
    try:
        pkv.paged_attention_decode(out, q, kc, vc, bt, cl, case["scale"], max_context_len=mcl,
                                   partition_size=partition_size, device_status=st)
    finally:
        ran = pkv.last_decode_engine()
        pkv.set_decode_engine("auto")
    torch.cuda.synchronize()
    if engine != "auto":
        assert ran == engine, (ran, engine)
    return out.to(torch.float64).cpu().numpy(), int(st.item()), pkv.last_decode_launches()


def oracle_decode(case, partition_size=0):
    return oracle.paged_attention(raw_np(case["q"]), raw_np(case["k_cache"]), raw_np(case["v_cache"]),
                                  case["dtype"], case["block_tables"], case["context_lens"],
                                  case["Hk"], case["scale"], partition_size=partition_size)


def max_err(a, b):
    return float(np.max(np.abs(a - b))) if a.size else 0.0


def ulp_bound(ref: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """One unit in the last place of `dtype` at the magnitude of ref."""
    mant = {torch.float16: 10, torch.bfloat16: 7}[dtype]
    tiny = {torch.float16: 2.0 ** -24, torch.bfloat16: 2.0 ** -133}[dtype]
    a = np.abs(ref)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    if dtype == torch.float16:
        e = np.maximum(e, -14)
    return np.maximum(2.0 ** (e - mant), tiny)


class SampledOracle:
    """Oracle copy of the blocks that a few sampled sequences touch.

    Built from the generator's initial cache values (read from the device
    before any library kernel writes to it), it then follows every step with
    the oracle's own copy-on-write copies and scatter, and answers attention
    for the sampled sequences only."""

    def __init__(self, state, seqs, steps_inputs):
        self.cfg = state.cfg
        self.seqs = list(seqs)
        blocks = set()
        for inp in steps_inputs:
            for s in self.seqs:
                L = int(inp.context_lens[s])
                nb = -(-L // self.cfg.block_size)
                blocks.update(int(b) for b in inp.block_tables[s][:nb])
            for a, b in inp.cow_pairs:
                if int(b) in blocks or int(a) in blocks:
                    blocks.update((int(a), int(b)))
        for inp in steps_inputs:           # sources of copies into tracked blocks
            for a, b in inp.cow_pairs:
                if int(b) in blocks:
                    blocks.add(int(a))
        self.blocks = np.array(sorted(blocks), dtype=np.int64)
        self.local = {int(b): i for i, b in enumerate(self.blocks)}
        idx = torch.as_tensor(self.blocks, device=state.k_cache.device)
        self.k = raw_np(state.k_cache.index_select(0, idx)).copy()
        self.v = raw_np(state.v_cache.index_select(0, idx)).copy()

    def _loc(self, b):
        return self.local.get(int(b), -1)

    def apply_step(self, inp, key, value):
        """Oracle copy-on-write copies and scatter for the tracked blocks."""
        bs = self.cfg.block_size
        pairs = [(self._loc(a), self._loc(b)) for a, b in inp.cow_pairs]
        pairs = [p for p in pairs if p[1] >= 0]
        if pairs:
            assert all(p[0] >= 0 for p in pairs)
            assert oracle.copy_blocks([self.k], [self.v], np.array(pairs, dtype=np.int64)) == 0
        slots = np.array([self._loc(sl // bs) * bs + sl % bs if self._loc(sl // bs) >= 0 else -1
                          for sl in inp.slot_mapping], dtype=np.int64)
        assert oracle.reshape_and_cache(raw_np(key), raw_np(value), self.k, self.v, slots) == 0

    def attention(self, inp, q):
        """fp64 oracle outputs [len(seqs), H, D] for the sampled sequences."""
        bs = self.cfg.block_size
        tables = np.full((len(self.seqs), inp.block_tables.shape[1]), -1, dtype=np.int32)
        lens = np.zeros(len(self.seqs), dtype=np.int32)
        for i, s in enumerate(self.seqs):
            L = int(inp.context_lens[s])
            lens[i] = L
            nb = -(-L // bs)
            tables[i, :nb] = [self._loc(b) for b in inp.block_tables[s][:nb]]
        qs = raw_np(q[self.seqs])
        out, st = oracle.paged_attention(qs, self.k, self.v, self.cfg.dtype, tables, lens,
                                         self.cfg.num_kv_heads,
                                         float(np.float32(self.cfg.softmax_scale)))
        assert st == 0
        return out
