"""GPU parity of paged_attention_decode against the CPU oracle.

Bars: max-abs error <= 1e-5 for fp32 K/V and <= 2e-3 for fp16/bf16 K/V with
fp32 output; fp16/bf16 output within one unit in the last place of the
oracle's value in that dtype; bit-identical results under physical block
permutation and prefix aliasing; L = 1 returns the value row exactly."""
import numpy as np
import pytest
import torch

from tests.gpu_support import TOL, gpu_decode, max_err, oracle_decode, ulp_bound
from tests.util import logical_kv, small_case

pytestmark = pytest.mark.gpu


def lens_for(bs):
    return (1, bs - 1, bs, bs + 1, 3 * bs + 5, 100, 511, 512, 513)


ENGINE_CASES = [(dt, e) for dt in ("f32", "f16", "bf16") for e in ("cuda_core", "tensor_core")
                if not (dt == "f32" and e == "tensor_core")]


@pytest.mark.parametrize("dtype,engine", ENGINE_CASES)
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_decode_matrix(dtype, engine, D, bs, G):
    lens = lens_for(bs)
    case = small_case(100 + D + bs + G, dtype=dtype, B=len(lens), H=2 * G, Hk=2, D=D, bs=bs,
                      lens=lens)
    ref, st = oracle_decode(case)
    assert st == 0
    for P in (0, 32, 4096):           # automatic, forced split (tiny partitions), forced single
        got, gst, launches = gpu_decode(case, partition_size=P, engine=engine)
        assert gst == 0
        assert launches == (2 if P == 32 else 1) or P == 0
        err = max_err(got, ref)
        assert err <= TOL[dtype], f"P={P} max err {err}"


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("engine", ["cuda_core", "tensor_core"])
def test_half_output_within_one_ulp(dtype, engine):
    """16-bit output is the fp32 result rounded to nearest even (bit-exact
    against the same call with fp32 output), so it lies within one 16-bit ulp
    of the oracle rounded to that type, plus the fp32 result's own error."""
    case = small_case(3, dtype=dtype, B=4, H=8, Hk=2, D=128, bs=16, lens=(7, 300, 64, 1000))
    ref, _ = oracle_decode(case)
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    rne = torch.from_numpy(ref).to(tdt).to(torch.float64).numpy()
    for P in (0, 64):
        got, st, _ = gpu_decode(case, partition_size=P, out_dtype=tdt, engine=engine)
        got32, st32, _ = gpu_decode(case, partition_size=P, engine=engine)
        assert st == 0 and st32 == 0
        np.testing.assert_array_equal(got, torch.from_numpy(got32).to(tdt).double().numpy())
        assert max_err(got32, ref) <= TOL[dtype]
        assert np.all(np.abs(got - rne) <= ulp_bound(ref, tdt) + np.abs(got32 - ref))


@pytest.mark.parametrize("engine", ["cuda_core", "tensor_core"])
def test_long_context_split_path(engine):
    lens = (4097, 16384 + 511, 9000)
    case = small_case(9, dtype="bf16", B=3, H=16, Hk=2, D=128, bs=16, lens=lens)
    ref, _ = oracle_decode(case)
    for P in (0, 512, 1024):
        got, st, launches = gpu_decode(case, partition_size=P, engine=engine)
        assert st == 0 and launches == 2
        assert max_err(got, ref) <= TOL["bf16"]


@pytest.mark.parametrize("engine", ["cuda_core", "tensor_core"])
@pytest.mark.parametrize("D", [64, 128])
def test_split_merge_over_many_rounds(D, engine):
    """Hundreds of 32-token partitions per context: the merge reads a
    context's slots in several rounds (eight warps, one slot lane each at
    head_dim 128 and two at 64, eight slots per lane per round), and keys
    carry a component along a fixed direction proportional to their
    position that every query shares, so the scores climb through the
    context and each round raises the running maxima.  An empty context and
    a one-partition one sit beside them."""
    lens = (5000, 1, 0, 2100, 40)
    case = small_case(77 + D, dtype="bf16", B=5, H=8, Hk=2, D=D, bs=16, lens=lens)
    bt = case["block_tables"]
    kc = case["k_cache"].float()
    u = torch.zeros(D)
    u[:8] = 1.0
    for s, L in enumerate(lens):
        for t in range(L):
            kc[int(bt[s, t // 16]), :, t % 16, :] += 0.01 * t * u
    case = dict(case, k_cache=kc.to(torch.bfloat16), q=(case["q"].float() + u).to(torch.bfloat16))
    ref, st = oracle_decode(case)
    assert st == 0
    for P in (32, 64):
        got, gst, launches = gpu_decode(case, partition_size=P, engine=engine)
        assert gst == 0 and launches == 2
        assert not got[2].any()
        assert max_err(got, ref) <= TOL["bf16"], f"P={P}"


@pytest.mark.parametrize("dtype,engine", [("f32", "cuda_core"), ("bf16", "cuda_core"),
                                          ("bf16", "tensor_core"), ("f16", "tensor_core")])
def test_empty_and_single_token(dtype, engine):
    case = small_case(4, dtype=dtype, B=4, H=8, Hk=2, D=64, bs=16, lens=(0, 1, 1, 0))
    for P in (0, 32):
        got, st, _ = gpu_decode(case, partition_size=P, engine=engine)
        assert st == 0
        assert not got[0].any() and not got[3].any()
        for s in (1, 2):
            _, V = logical_kv(case, s)
            # exactly v_0 of each query head's kv head (head h reads kv head h // 4)
            np.testing.assert_array_equal(got[s], np.repeat(V[0], 4, axis=0))


@pytest.mark.parametrize("engine", ["cuda_core", "tensor_core"])
def test_permutation_is_bit_exact(engine):
    case = small_case(5, dtype="bf16", B=3, H=8, Hk=1, D=128, bs=16, lens=(70, 513, 1200))
    base, _, _ = gpu_decode(case, partition_size=512, engine=engine)
    NB = case["k_cache"].shape[0]
    perm = torch.randperm(NB, generator=torch.Generator().manual_seed(1))
    moved = dict(case)
    moved["k_cache"] = torch.empty_like(case["k_cache"]); moved["k_cache"][perm] = case["k_cache"]
    moved["v_cache"] = torch.empty_like(case["v_cache"]); moved["v_cache"][perm] = case["v_cache"]
    t = case["block_tables"]
    moved["block_tables"] = np.where(t >= 0, perm.numpy()[np.maximum(t, 0)], -1).astype(np.int32)
    got, st, _ = gpu_decode(moved, partition_size=512, engine=engine)
    assert st == 0
    np.testing.assert_array_equal(got, base)


@pytest.mark.parametrize("engine", ["cuda_core", "tensor_core"])
def test_prefix_aliasing_is_bit_exact(engine):
    g = torch.Generator().manual_seed(6)
    bs, Hk, H, D = 16, 2, 8, 128
    kc = torch.randn(16, Hk, bs, D, generator=g).to(torch.bfloat16)
    vc = torch.randn(16, Hk, bs, D, generator=g).to(torch.bfloat16)
    kc[4:8] = kc[0:4]; vc[4:8] = vc[0:4]
    q = torch.randn(1, H, D, generator=g).to(torch.bfloat16).repeat(2, 1, 1)
    base = dict(q=q, k_cache=kc, v_cache=vc, dtype="bf16", bs=bs, Hk=Hk, scale=0.088388,
                context_lens=np.array([4 * bs + 3, 4 * bs + 3], np.int32))
    dup = dict(base, block_tables=np.array([[0, 1, 2, 3, 8], [4, 5, 6, 7, 8]], np.int32))
    ali = dict(base, block_tables=np.array([[0, 1, 2, 3, 8], [0, 1, 2, 3, 8]], np.int32))
    a, _, _ = gpu_decode(dup, engine=engine)
    b, _, _ = gpu_decode(ali, engine=engine)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(a[0], a[1])


@pytest.mark.parametrize("engine", ["cuda_core", "tensor_core"])
def test_bad_block_and_length_are_reported(engine):
    import paged_kv_cache_311_gb300 as pkv
    case = small_case(7, dtype="f16", B=3, H=4, Hk=2, D=128, bs=16, lens=(40, 40, 40))
    # the unaffected sequence must match the clean run on the same path bit for bit
    good = {P: gpu_decode(case, partition_size=P, engine=engine)[0] for P in (0, 32)}
    bad = dict(case)
    t = case["block_tables"].copy()
    t[1, 2] = case["k_cache"].shape[0] + 5
    bad["block_tables"] = t
    for P in (0, 32):
        got, st, _ = gpu_decode(bad, partition_size=P, engine=engine)
        assert st & pkv.DEV_BAD_BLOCK
        assert not got[1].any()
        np.testing.assert_array_equal(got[0], good[P][0])
    lens = case["context_lens"].copy()
    lens[2] = 41                                # beyond max_context_len passed below
    bl = dict(case, context_lens=lens)
    for P in (0, 32):
        got, st, _ = gpu_decode(bl, partition_size=P, max_context_len=40, engine=engine)
        assert st & pkv.DEV_BAD_CONTEXT_LEN
        assert not got[2].any()
        np.testing.assert_array_equal(got[0], good[P][0])


def test_host_validation_rejects_bad_arguments():
    import paged_kv_cache_311_gb300 as pkv
    case = small_case(8, dtype="f16", B=2, H=4, Hk=2, D=128, bs=16, lens=(5, 6))
    with pytest.raises(pkv.PkvError) as e:
        gpu_decode(case, partition_size=48)     # not a multiple of 32
    assert e.value.status == -1
    odd = small_case(8, dtype="f16", B=2, H=6, Hk=2, D=128, bs=16, lens=(5, 6))   # G = 3
    with pytest.raises(pkv.PkvError) as e:
        gpu_decode(odd)
    assert e.value.status == -2
