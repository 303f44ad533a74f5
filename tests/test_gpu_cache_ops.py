"""GPU reshape_and_cache and copy_blocks: bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from tests.util import DT, raw_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("D,bs,Hk", [(64, 16, 4), (128, 8, 8), (128, 32, 40)])
def test_reshape_and_cache_bit_exact(dtype, D, bs, Hk):
    import paged_kv_cache_311_gb300 as pkv
    g = torch.Generator().manual_seed(D + bs + Hk)
    NB, T = 50, 300
    kc = torch.randn(NB, Hk, bs, D, generator=g).to(DT[dtype])
    vc = torch.randn(NB, Hk, bs, D, generator=g).to(DT[dtype])
    key = torch.randn(T, Hk, D, generator=g).to(DT[dtype])
    val = torch.randn(T, Hk, D, generator=g).to(DT[dtype])
    slots = torch.randperm(NB * bs, generator=g)[:T].to(torch.int64)
    slots[::37] = -1                                 # padding tokens
    k_ref, v_ref = raw_np(kc).copy(), raw_np(vc).copy()
    assert oracle.reshape_and_cache(raw_np(key), raw_np(val), k_ref, v_ref, slots.numpy()) == 0
    kd, vd = kc.cuda(), vc.cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.reshape_and_cache(key.cuda(), val.cuda(), kd, vd, slots.cuda(), device_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(raw_np(kd).view(np.uint8), k_ref.view(np.uint8))
    assert np.array_equal(raw_np(vd).view(np.uint8), v_ref.view(np.uint8))


def test_reshape_and_cache_bad_slot_is_skipped_and_reported():
    import paged_kv_cache_311_gb300 as pkv
    NB, Hk, bs, D = 4, 2, 16, 64
    kc = torch.zeros(NB, Hk, bs, D, device="cuda")
    vc = torch.zeros_like(kc)
    key = torch.ones(3, Hk, D, device="cuda")
    slots = torch.tensor([0, NB * bs, 5], dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.reshape_and_cache(key, key, kc, vc, slots, device_status=st)
    torch.cuda.synchronize()
    assert st.item() == pkv.DEV_BAD_SLOT
    assert kc[0, :, 0].eq(1).all() and kc[0, :, 5].eq(1).all() and kc.sum().item() == 2 * Hk * D


def test_reshape_and_cache_empty_is_a_no_op():
    import paged_kv_cache_311_gb300 as pkv
    kc = torch.zeros(2, 1, 16, 64, device="cuda")
    pkv.reshape_and_cache(torch.zeros(0, 1, 64, device="cuda"), torch.zeros(0, 1, 64, device="cuda"),
                          kc, kc.clone(), torch.zeros(0, dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert kc.abs().sum().item() == 0


@pytest.mark.parametrize("layers", [1, 3, 130])
def test_copy_blocks_bit_exact(layers):
    import paged_kv_cache_311_gb300 as pkv
    g = torch.Generator().manual_seed(layers)
    NB, shape = 24, (8, 16, 128)
    ks = [torch.randn((NB,) + shape, generator=g).to(torch.bfloat16) for _ in range(layers)]
    vs = [torch.randn((NB,) + shape, generator=g).to(torch.bfloat16) for _ in range(layers)]
    pairs = np.array([[1, 10], [2, 11], [1, 12], [5, 20]], dtype=np.int64)
    ref_k = [raw_np(k).copy() for k in ks]
    ref_v = [raw_np(v).copy() for v in vs]
    assert oracle.copy_blocks(ref_k, ref_v, pairs) == 0
    kd = [k.cuda() for k in ks]
    vd = [v.cuda() for v in vs]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.copy_blocks(kd, vd, torch.as_tensor(pairs).cuda(), device_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    for l in range(layers):
        assert np.array_equal(raw_np(kd[l]), ref_k[l])
        assert np.array_equal(raw_np(vd[l]), ref_v[l])


def test_copy_blocks_bad_pair_is_skipped_and_reported():
    import paged_kv_cache_311_gb300 as pkv
    kc = torch.arange(4 * 256, dtype=torch.float32, device="cuda").view(4, 1, 4, 64)
    vc = kc.clone()
    before = kc.clone()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pairs = torch.tensor([[0, 4], [1, 2]], dtype=torch.int64, device="cuda")
    pkv.copy_blocks([kc], [vc], pairs, device_status=st)
    torch.cuda.synchronize()
    assert st.item() == pkv.DEV_BAD_BLOCK
    assert torch.equal(kc[2], before[1]) and torch.equal(kc[0], before[0]) and torch.equal(kc[3], before[3])


def _swap_case(seed, layers, NB, NH, Hk, bs, D, dtype):
    g = torch.Generator().manual_seed(seed)
    gk = [torch.randn(NB, Hk, bs, D, generator=g).to(DT[dtype]) for _ in range(layers)]
    gv = [torch.randn(NB, Hk, bs, D, generator=g).to(DT[dtype]) for _ in range(layers)]
    hk = [torch.zeros(NH, Hk, bs, D, dtype=DT[dtype]).pin_memory() for _ in range(layers)]
    hv = [torch.zeros(NH, Hk, bs, D, dtype=DT[dtype]).pin_memory() for _ in range(layers)]
    return gk, gv, hk, hv


def _bytes(t):
    return raw_np(t.cpu()).view(np.uint8)


@pytest.mark.parametrize("dtype,Hk,bs,D,layers", [("bf16", 8, 16, 128, 3), ("f16", 4, 8, 64, 1),
                                                  ("f32", 2, 32, 64, 2)])
def test_swap_blocks_round_trip_bit_exact(dtype, Hk, bs, D, layers):
    """Swap-out writes each pair's GPU block into its host block, bit for bit
    as the oracle's copy; after the GPU blocks were reused, swap-in puts them
    back."""
    import paged_kv_cache_311_gb300 as pkv
    NB, NH = 64, 40
    gk, gv, hk, hv = _swap_case(7 + Hk, layers, NB, NH, Hk, bs, D, dtype)
    rng = np.random.default_rng(Hk)
    pairs = np.stack([rng.permutation(NB)[:30], rng.permutation(NH)[:30]], axis=1).astype(np.int64)
    ref_hk = [raw_np(h).copy() for h in hk]; ref_hv = [raw_np(h).copy() for h in hv]
    ref_gk = [raw_np(x).copy() for x in gk]; ref_gv = [raw_np(x).copy() for x in gv]
    assert oracle.swap_blocks(ref_gk, ref_gv, ref_hk, ref_hv, pairs, 0) == 0
    dk = [x.cuda() for x in gk]; dv = [x.cuda() for x in gv]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dp = torch.from_numpy(pairs).cuda()
    pkv.swap_blocks(dk, dv, hk, hv, dp, pkv.SWAP_OUT, device_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    for l in range(layers):
        assert np.array_equal(_bytes(hk[l]), ref_hk[l].view(np.uint8))
        assert np.array_equal(_bytes(hv[l]), ref_hv[l].view(np.uint8))
        dk[l][dp[:, 0]] = 0      # the blocks are reused while the sequence is out
        dv[l][dp[:, 0]] = 0
    pkv.swap_blocks(dk, dv, hk, hv, dp, pkv.SWAP_IN, device_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    for l in range(layers):
        assert np.array_equal(_bytes(dk[l]), raw_np(gk[l]).view(np.uint8))
        assert np.array_equal(_bytes(dv[l]), raw_np(gv[l]).view(np.uint8))


def test_swap_blocks_many_small_blocks_in_one_launch():
    """The small-block case the pages call costly for swapping (many small
    transfers): 2,000 blocks of 8 rows move in one launch, bit-exact."""
    import paged_kv_cache_311_gb300 as pkv
    NB, NH = 4096, 2048
    gk, gv, hk, hv = _swap_case(3, 1, NB, NH, 8, 8, 64, "bf16")
    pairs = np.stack([np.random.default_rng(1).permutation(NB)[:2000], np.arange(2000)], 1)
    dp = torch.from_numpy(pairs.astype(np.int64)).cuda()
    dk, dv = [gk[0].cuda()], [gv[0].cuda()]
    pkv.swap_blocks(dk, dv, hk, hv, dp, pkv.SWAP_OUT)
    torch.cuda.synchronize()
    assert np.array_equal(_bytes(hk[0])[:2000], raw_np(gk[0]).view(np.uint8)[pairs[:, 0]])
    assert np.array_equal(_bytes(hv[0])[:2000], raw_np(gv[0]).view(np.uint8)[pairs[:, 0]])


def test_swap_blocks_bad_pair_and_unpinned_host():
    import paged_kv_cache_311_gb300 as pkv
    gk, gv, hk, hv = _swap_case(5, 1, 8, 4, 2, 16, 64, "f16")
    dk, dv = [gk[0].cuda()], [gv[0].cuda()]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dp = torch.tensor([[1, 0], [8, 1], [2, 4], [3, 2]], dtype=torch.int64, device="cuda")
    pkv.swap_blocks(dk, dv, hk, hv, dp, pkv.SWAP_OUT, device_status=st)
    torch.cuda.synchronize()
    assert st.item() & pkv.DEV_BAD_BLOCK
    assert np.array_equal(_bytes(hk[0])[0], raw_np(gk[0]).view(np.uint8)[1])
    assert np.array_equal(_bytes(hk[0])[2], raw_np(gk[0]).view(np.uint8)[3])
    assert not _bytes(hk[0])[1].any()                    # the (8, 1) pair was skipped
    with pytest.raises(ValueError):
        pkv.swap_blocks(dk, dv, [torch.zeros_like(hk[0])], hv, dp, pkv.SWAP_OUT)
