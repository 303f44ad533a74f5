"""Helpers shared by the tests: raw-bit views and small seeded cases."""
from __future__ import annotations

import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def raw_np(t: torch.Tensor) -> np.ndarray:
    """Host numpy view of a tensor's raw elements (bf16 comes back as uint16 bits)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


def read_golden(name: str):
    rows, meta = [], {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if not parts[0].lstrip("-").isdigit():
                meta[parts[0]] = parts[1]
                continue
            rows.append([int(x) for x in parts])
    return meta, rows


DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def small_case(seed: int, *, dtype="f32", B=3, H=4, Hk=2, D=64, bs=16, lens=(1, 17, 40),
               pool=None, permute=True, device="cpu"):
    """A seeded paged-cache case: q [B,H,D], caches [NB,Hk,bs,D], int32 tables/lens.

    Blocks are placed by a seeded permutation of the pool (or in order when
    ``permute`` is False, giving the identity layout)."""
    g = torch.Generator().manual_seed(seed)
    lens = list(lens)
    nblk = [-(-L // bs) for L in lens]
    MB = max(max(nblk), 1)
    NB = pool if pool is not None else max(sum(nblk) + 3, 4)
    order = torch.randperm(NB, generator=g).tolist() if permute else list(range(NB))
    tables = np.full((B, MB), -1, dtype=np.int32)
    k = 0
    for s in range(B):
        for j in range(nblk[s]):
            tables[s, j] = order[k]
            k += 1
    q = torch.randn(B, H, D, generator=g).to(DT[dtype])
    kc = torch.randn(NB, Hk, bs, D, generator=g).to(DT[dtype])
    vc = torch.randn(NB, Hk, bs, D, generator=g).to(DT[dtype])
    return dict(q=q.to(device), k_cache=kc.to(device), v_cache=vc.to(device), block_tables=tables,
                context_lens=np.array(lens, dtype=np.int32), dtype=dtype, bs=bs, Hk=Hk,
                scale=float(np.float32(1.0 / np.sqrt(D))))


def logical_kv(case, s: int):
    """Gather sequence s's logical K, V [L, Hk, D] in fp64 with torch indexing."""
    L = int(case["context_lens"][s])
    bs = case["bs"]
    pos = np.arange(L)
    blocks = case["block_tables"][s][pos // bs]
    offs = pos % bs
    kc = case["k_cache"].cpu().to(torch.float64)
    vc = case["v_cache"].cpu().to(torch.float64)
    bi = torch.as_tensor(blocks, dtype=torch.long)
    oi = torch.as_tensor(offs, dtype=torch.long)
    return kc[bi, :, oi, :].numpy(), vc[bi, :, oi, :].numpy()
