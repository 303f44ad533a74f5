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
