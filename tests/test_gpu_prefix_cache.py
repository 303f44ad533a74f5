"""Prefix caching and parallel sampling end to end on the GPU, at full size.

The block tables, prefill slots, decode slots and copy-on-write pairs come
from the product's block pool (DecodeBatch over BlockPool), checked call by
call against the oracle's prefix-cache model (tests/pool_lockstep.py).  The
GPU then runs what a serving step runs -- the prefill scatter of every
request's uncached tokens, and per decode step the copy-on-write copies, the
scatter of the new tokens, the shared-prefix decode (both kernels) and the
per-sequence decode -- and every sequence's output is compared with the
oracle, which applies its own scatter and copies to a host copy of the cache
and attends through the same tables.  At the end both caches agree bit for
bit.

Workloads follow the page "PagedAttention: Efficient LLM Serving with vLLM",
"Advanced Features": 256 requests over 4 cached system prompts of 1024-2048
tokens plus 32-256 of their own (Prefix Caching: the first request of a prompt
computes its blocks, all later ones reuse them), and 32 prompts of 256-1024
tokens forked into 6 samples each (KV-Cache Sharing: only the divergent
tokens get new blocks); bf16, 32 query / 8 kv heads, head_dim 128, block 16.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_311_gb300 as pkv
from tests.gpu_support import TOL, max_err
from tests.pool_lockstep import (Lockstep, build_sampling, build_system_prompt, sampling_prompts,
                                 system_prompt_requests)
from tests.util import raw_np

pytestmark = pytest.mark.gpu

H, HK, D, BS = 32, 8, 128, 16
SCALE = float(np.float32(1.0 / np.sqrt(D)))


def _bf16(gen, *shape):
    return torch.randn(*shape, generator=gen).to(torch.bfloat16)


def _run(ls, B, prefill_slots, steps, seed):
    dev = torch.device("cuda")
    NB = ls.pool.num_blocks
    gen = torch.Generator().manual_seed(seed)
    kc = torch.zeros((NB, HK, BS, D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    okc = np.zeros((NB, HK, BS, D), np.uint16)
    ovc = np.zeros_like(okc)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    nthreads = os.cpu_count() or 1

    # prefill: every request's tokens that the prefix cache did not hold
    slots = np.concatenate(prefill_slots).astype(np.int64)
    k, v = _bf16(gen, slots.size, HK, D), _bf16(gen, slots.size, HK, D)
    pkv.reshape_and_cache(k.to(dev), v.to(dev), kc, vc, torch.from_numpy(slots).to(dev),
                          device_status=st)
    assert oracle.reshape_and_cache(raw_np(k), raw_np(v), okc, ovc, slots) == 0

    worst = {}
    for t in range(steps):
        slots, pairs = ls.step(B)
        q = _bf16(gen, B, H, D)
        k, v = _bf16(gen, B, HK, D), _bf16(gen, B, HK, D)
        if pairs.shape[0]:
            pkv.copy_blocks([kc], [vc], torch.from_numpy(pairs).to(dev), device_status=st)
            assert oracle.copy_blocks([okc], [ovc], pairs) == 0
        pkv.reshape_and_cache(k.to(dev), v.to(dev), kc, vc, torch.from_numpy(slots).to(dev),
                              device_status=st)
        assert oracle.reshape_and_cache(raw_np(k), raw_np(v), okc, ovc, slots) == 0

        tables = ls.batch.tables[:B].copy()
        lens = ls.batch.lens[:B].copy()
        qd = q.to(dev)
        bt, cl = torch.from_numpy(tables).to(dev), torch.from_numpy(lens).to(dev)
        outs = {}
        plan = pkv.plan_shared_prefix(tables, lens, H, HK, D, BS, int(lens.max()), 0)
        plan_dev = plan.to(dev)
        for engine in ("auto", "tcgen05"):
            pkv.set_decode_engine(engine)
            try:
                o = torch.full((B, H, D), float("nan"), dtype=torch.float32, device=dev)
                pkv.paged_attention_decode_shared(o, qd, kc, vc, bt, cl, SCALE, plan, plan_dev,
                                                  max_context_len=int(lens.max()), device_status=st)
                outs["shared_" + pkv.last_decode_engine()] = o
            finally:
                pkv.set_decode_engine("auto")
        o = torch.full((B, H, D), float("nan"), dtype=torch.float32, device=dev)
        pkv.paged_attention_decode(o, qd, kc, vc, bt, cl, SCALE, max_context_len=int(lens.max()),
                                   device_status=st)
        outs["per_sequence"] = o
        torch.cuda.synchronize()
        assert st.item() == 0
        ref, ost = oracle.paged_attention(raw_np(q), okc, ovc, "bf16", tables, lens, HK, SCALE,
                                          nthreads=nthreads)
        assert ost == 0
        for name, o in outs.items():
            e = max_err(o.double().cpu().numpy(), ref)
            worst[name] = max(worst.get(name, 0.0), e)
            assert e <= TOL["bf16"], (t, name, e)
    assert np.array_equal(raw_np(kc), okc) and np.array_equal(raw_np(vc), ovc)
    assert set(worst) == {"shared_tensor_core", "shared_tcgen05", "per_sequence"}
    return worst


def test_system_prompt_requests_on_cached_prefix_blocks():
    B, steps = 256, 4
    reqs, prompts = system_prompt_requests(3111, B, 4, (1024, 2048), (32, 256))
    ls = Lockstep(8192, BS, B, 160)
    pre = build_system_prompt(ls, reqs)
    # each prompt's first request computes it; the other 252 reuse its full blocks
    assert [c for _, c in pre] == [0] * 4 + [len(prompts[i % 4]) // BS * BS for i in range(4, B)]
    for p in range(4):
        first = ls.batch.tables[p, : len(prompts[p]) // BS]
        assert (first >= 0).all()
        assert ls.pool.refcount(int(first[0])) == B // 4
    _run(ls, B, [s for s, _ in pre], steps, seed=3112)
    ls.check_holders()


def test_forked_samples_share_their_prompt_until_they_diverge():
    S, P, steps = 6, 32, 4
    prompts = sampling_prompts(3113, P, (256, 1024))
    ls = Lockstep(4096, BS, P * S, 80)
    pre = build_sampling(ls, prompts, S)
    before = ls.pool.available()
    worst = _run(ls, P * S, [s for s, _ in pre], steps, seed=3114)
    # only the divergent tokens took new blocks: each prompt's full blocks stay
    # shared, each sample ends up owning the blocks past them (a copy of the
    # shared partial block for five of the six samples, the original for one)
    want = sum(p.size // BS + S * (-(-(p.size + steps) // BS) - p.size // BS) - -(-p.size // BS)
               for p in prompts)
    assert before - ls.pool.available() == want
    for p in range(P):
        head = ls.batch.tables[p * S, : prompts[p].size // BS]
        for k in range(1, S):
            assert (ls.batch.tables[p * S + k, : head.size] == head).all()
    ls.check_holders()
    assert worst["shared_tensor_core"] <= TOL["bf16"]
