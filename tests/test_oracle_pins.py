"""Pins for the CPU oracle: facts that the pages and the mathematics fix.

Each test compares the oracle with something other than itself:
  * the worked block-count and page-table examples of the page
    "PagedAttention: Efficient LLM Serving with vLLM" (tests/golden/),
  * numpy / torch dtype conversions for the fp16 and bf16 decoders,
  * torch's scaled_dot_product_attention in fp64 (a library routine) over the
    logical tokens gathered with torch indexing,
  * closed forms (one token, zero query, identical keys, one dominant key),
  * the paging invariants the pages state: blocks may sit anywhere (physical
    permutation), shared prefix blocks equal duplicated ones, block size only
    trades overhead for waste,
  * the exact log-sum-exp regrouping of the split-context merge,
  * numpy fancy-index scatter and slice copies for the cache scatter and the
    copy-on-write block copy.
"""
import numpy as np
import pytest
import torch

from tests.util import f64, logical_kv, raw_np, read_golden, small_case


def run_oracle(oracle, case, partition_size=0, nthreads=1, tables=None, k_cache=None, v_cache=None):
    return oracle.paged_attention(
        raw_np(case["q"]), raw_np(case["k_cache"] if k_cache is None else k_cache),
        raw_np(case["v_cache"] if v_cache is None else v_cache), case["dtype"],
        case["block_tables"] if tables is None else tables, case["context_lens"], case["Hk"],
        case["scale"], partition_size=partition_size, nthreads=nthreads)


def sdpa_reference(case):
    """torch SDPA (fp64, CPU) over each sequence's logical tokens."""
    q = f64(case["q"])
    B, H, D = q.shape
    G = H // case["Hk"]
    out = np.zeros((B, H, D))
    for s in range(B):
        L = int(case["context_lens"][s])
        if L == 0:
            continue
        K, V = logical_kv(case, s)
        Kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
        Vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
        qt = torch.from_numpy(q[s])[None, :, None, :]
        o = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, scale=case["scale"])
        out[s] = o[0, :, 0, :].numpy()
    return out


# --------------------------------------------------------------- blocks
def test_worked_example_block_count(oracle_lib):
    from oracle.block_manager import OracleBlockManager
    _, rows = read_golden("worked_example_blocks.txt")
    for tokens, bs, blocks, slots, unused in rows:
        assert oracle_lib.blocks_for_tokens(tokens, bs) == blocks
        bm = OracleBlockManager(num_blocks=64, block_size=bs)
        bm.add_sequence(0, tokens)
        assert len(bm.tables[0]) == blocks
        assert bm.allocated_slots(0) == slots
        assert bm.unused_slots(0) == unused


def test_blocks_on_demand():
    from oracle.block_manager import OracleBlockManager, blocks_for_tokens
    bm = OracleBlockManager(num_blocks=32, block_size=16)
    bm.add_sequence(0, 1)
    for n in range(2, 200):
        bm.append_token(0)
        assert len(bm.tables[0]) == blocks_for_tokens(n, 16) == -(-n // 16)
    assert len(set(bm.tables[0])) == len(bm.tables[0])


def test_blocks_return_when_their_last_sharer_frees():
    """A finished sequence's blocks go back to the pool; a block it shares
    with a fork stays held until the fork finishes too (reference counts;
    "Advanced Features", KV-Cache Sharing)."""
    from oracle.block_manager import OracleBlockManager
    bm = OracleBlockManager(num_blocks=16, block_size=16)
    bm.add_sequence(0, 40)          # blocks for tokens 0-15, 16-31, 32-39
    bm.fork(0, 1)
    bm.append_token(1)              # the shared partial block is copied for the fork
    assert len(bm.free) == 16 - 4
    bm.free_sequence(0)             # the two full blocks stay with the fork
    assert len(bm.free) == 16 - 3
    bm.free_sequence(1)
    assert len(bm.free) == 16 and all(r == 0 for r in bm.refcount)


def test_page_table_example(oracle_lib):
    """Logical block 0 -> physical 47, logical 1 -> physical 123: with a single
    dominant key at logical position p the output is exactly the V row stored
    at block table[p // bs], offset p % bs."""
    meta, rows = read_golden("page_table_example.txt")
    bs = int(meta["block_size"])
    table = np.array([[phys for _, phys in sorted(rows)]], dtype=np.int32)
    NB, D = 128, 8
    kc = np.zeros((NB, 1, bs, D), dtype=np.float32)
    vc = np.zeros((NB, 1, bs, D), dtype=np.float32)
    for b in range(NB):
        for o in range(bs):
            vc[b, 0, o, :] = b * 1000 + o      # V row names its own location
    for p in (0, 5, 15, 16, 17, 31):
        k = kc.copy()
        phys, off = table[0, p // bs], p % bs
        k[phys, 0, off, 0] = 1.0               # the only key aligned with q
        q = np.zeros((1, 1, D), dtype=np.float32)
        q[0, 0, 0] = 1000.0
        out, st = oracle_lib.paged_attention(q, k, vc, "f32", table, np.array([2 * bs], np.int32),
                                             1, 1.0)
        assert st == 0
        np.testing.assert_array_equal(out[0, 0], np.full(D, phys * 1000 + off, dtype=np.float64))


# ------------------------------------------------------------ decoders
def test_f16_decoder_matches_numpy(oracle_lib):
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_lib.f16_to_f64(int(b)) for b in bits])
    finite = np.isfinite(ref)
    np.testing.assert_array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_bf16_decoder_matches_torch(oracle_lib):
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle_lib.bf16_to_f64(int(b)) for b in bits])
    finite = np.isfinite(ref)
    np.testing.assert_array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


# ----------------------------------------------------- library attention
CASES = [
    dict(dtype="f32", B=3, H=4, Hk=4, D=64, bs=16, lens=(1, 17, 100)),
    dict(dtype="f16", B=3, H=8, Hk=2, D=128, bs=8, lens=(9, 64, 33)),
    dict(dtype="bf16", B=4, H=8, Hk=1, D=64, bs=32, lens=(31, 32, 33, 70)),
    dict(dtype="bf16", B=2, H=6, Hk=3, D=128, bs=16, lens=(513, 250)),
]


@pytest.mark.parametrize("kw", CASES)
def test_paged_matches_library_sdpa(oracle_lib, kw):
    case = small_case(7, **kw)
    out, st = run_oracle(oracle_lib, case)
    assert st == 0
    np.testing.assert_allclose(out, sdpa_reference(case), rtol=0, atol=1e-12)


def test_contiguous_matches_library_sdpa(oracle_lib):
    g = torch.Generator().manual_seed(3)
    L, H, Hk, D = 37, 8, 2, 64
    q = torch.randn(H, D, generator=g, dtype=torch.float64)
    K = torch.randn(L, Hk, D, generator=g, dtype=torch.float64)
    V = torch.randn(L, Hk, D, generator=g, dtype=torch.float64)
    got = oracle_lib.contiguous_attention(q.numpy(), K.numpy(), V.numpy(), 0.125)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q[None, :, None, :], K.permute(1, 0, 2).repeat_interleave(4, 0)[None],
        V.permute(1, 0, 2).repeat_interleave(4, 0)[None], scale=0.125)[0, :, 0, :]
    np.testing.assert_allclose(got, ref.numpy(), rtol=0, atol=1e-13)


# ------------------------------------------------------------ invariants
def test_permutation_invariance_bit_exact(oracle_lib):
    case = small_case(11, dtype="bf16", B=3, H=4, Hk=2, D=64, bs=16, lens=(5, 48, 77))
    base, _ = run_oracle(oracle_lib, case)
    NB = case["k_cache"].shape[0]
    perm = np.random.default_rng(5).permutation(NB)      # new home of each block
    kc = torch.empty_like(case["k_cache"]); vc = torch.empty_like(case["v_cache"])
    kc[torch.as_tensor(perm)] = case["k_cache"]; vc[torch.as_tensor(perm)] = case["v_cache"]
    tables = np.where(case["block_tables"] >= 0, perm[np.maximum(case["block_tables"], 0)], -1)
    moved, _ = run_oracle(oracle_lib, case, tables=tables.astype(np.int32), k_cache=kc, v_cache=vc)
    np.testing.assert_array_equal(moved, base)


def test_aliasing_equals_duplication_bit_exact(oracle_lib):
    """Two sequences sharing prefix blocks through their tables give the same
    outputs as the same tokens stored twice."""
    g = torch.Generator().manual_seed(2)
    bs, Hk, H, D = 16, 2, 4, 64
    prefix_blocks, tail = 3, 5
    NB = 2 * prefix_blocks + 2 + 2
    kc = torch.randn(NB, Hk, bs, D, generator=g).to(torch.float16)
    vc = torch.randn(NB, Hk, bs, D, generator=g).to(torch.float16)
    q = torch.randn(2, H, D, generator=g).to(torch.float16)
    # duplicated: seq0 uses blocks 0..2 + 6, seq1 uses copies 3..5 + 7
    kd, vd = kc.clone(), vc.clone()
    kd[3:6] = kd[0:3]; vd[3:6] = vd[0:3]
    dup = np.array([[0, 1, 2, 6], [3, 4, 5, 7]], dtype=np.int32)
    ali = np.array([[0, 1, 2, 6], [0, 1, 2, 7]], dtype=np.int32)
    lens = np.array([prefix_blocks * bs + tail] * 2, dtype=np.int32)
    a, _ = oracle_lib.paged_attention(raw_np(q), raw_np(kd), raw_np(vd), "f16", dup, lens, Hk, 0.125)
    b, _ = oracle_lib.paged_attention(raw_np(q), raw_np(kd), raw_np(vd), "f16", ali, lens, Hk, 0.125)
    np.testing.assert_array_equal(a, b)


def _relayout(K, V, bs, NB, rng):
    """Store logical K, V [L, Hk, D] into a fresh pool with block size bs."""
    L, Hk, D = K.shape
    nb = -(-L // bs)
    order = rng.permutation(NB)[:nb]
    kc = np.zeros((NB, Hk, bs, D), dtype=K.dtype); vc = np.zeros_like(kc)
    for i in range(L):
        kc[order[i // bs], :, i % bs, :] = K[i]; vc[order[i // bs], :, i % bs, :] = V[i]
    return kc, vc, order.astype(np.int32)


def test_block_size_invariance_bit_exact(oracle_lib):
    rng = np.random.default_rng(9)
    L, Hk, H, D = 90, 2, 8, 64
    K = rng.standard_normal((L, Hk, D)).astype(np.float32)
    V = rng.standard_normal((L, Hk, D)).astype(np.float32)
    q = rng.standard_normal((1, H, D)).astype(np.float32)
    outs = []
    for bs in (8, 16, 32):
        kc, vc, order = _relayout(K, V, bs, 40, rng)
        out, st = oracle_lib.paged_attention(q, kc, vc, "f32", order[None, :], np.array([L], np.int32),
                                             Hk, 0.125)
        assert st == 0
        outs.append(out)
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])


def test_gqa_equals_mha_with_repeated_heads(oracle_lib):
    case = small_case(4, dtype="f16", B=2, H=8, Hk=2, D=64, bs=16, lens=(20, 51))
    gqa, _ = run_oracle(oracle_lib, case)
    G = 4
    rep = dict(case)
    rep["k_cache"] = case["k_cache"].repeat_interleave(G, dim=1)
    rep["v_cache"] = case["v_cache"].repeat_interleave(G, dim=1)
    rep["Hk"] = 8
    mha, _ = run_oracle(oracle_lib, rep)
    np.testing.assert_array_equal(gqa, mha)


# ------------------------------------------------------------ closed forms
def test_single_token_returns_its_value_row(oracle_lib):
    case = small_case(5, dtype="bf16", B=3, H=4, Hk=4, D=64, bs=16, lens=(1, 1, 1))
    out, _ = run_oracle(oracle_lib, case)
    for s in range(3):
        _, V = logical_kv(case, s)
        np.testing.assert_array_equal(out[s], V[0])


def test_zero_query_gives_mean_of_values(oracle_lib):
    case = small_case(6, dtype="f32", B=2, H=2, Hk=2, D=64, bs=8, lens=(13, 40))
    case["q"] = torch.zeros_like(case["q"])
    out, _ = run_oracle(oracle_lib, case)
    for s in range(2):
        _, V = logical_kv(case, s)
        np.testing.assert_allclose(out[s], V.mean(axis=0), rtol=0, atol=1e-14)


def test_identical_keys_give_mean_of_values(oracle_lib):
    case = small_case(8, dtype="f32", B=1, H=2, Hk=1, D=64, bs=16, lens=(45,))
    kc = case["k_cache"].clone()
    kc[:] = kc[0, 0, 0]
    out, _ = run_oracle(oracle_lib, case, k_cache=kc)
    _, V = logical_kv(case, 0)
    np.testing.assert_allclose(out[0], np.repeat(V.mean(axis=0), 2, axis=0), rtol=0, atol=1e-14)


def test_dominant_key_selects_its_value(oracle_lib):
    case = small_case(10, dtype="f32", B=1, H=1, Hk=1, D=64, bs=16, lens=(60,))
    K, V = logical_kv(case, 0)
    q = torch.zeros_like(case["q"])
    q[0, 0, 0] = 1.0
    kc = case["k_cache"].clone()
    kc[..., 0] = 0.0
    target = 37
    phys, off = case["block_tables"][0, target // 16], target % 16
    kc[phys, 0, off, 0] = 800.0                 # z gap = 100 >= 60 above every other key
    case["q"] = q
    out, _ = run_oracle(oracle_lib, case, k_cache=kc)
    np.testing.assert_allclose(out[0, 0], V[target, 0], rtol=0, atol=1e-20 + 1e-40)


# ---------------------------------------------------- split-context merge
@pytest.mark.parametrize("P", [1, 7, 16, 64, 512])
def test_partitioned_merge_equals_single_pass(oracle_lib, P):
    case = small_case(12, dtype="bf16", B=3, H=8, Hk=2, D=128, bs=16, lens=(1, 300, 1025))
    a, _ = run_oracle(oracle_lib, case)
    b, _ = run_oracle(oracle_lib, case, partition_size=P)
    np.testing.assert_allclose(b, a, rtol=0, atol=1e-13)


def test_threads_bit_exact(oracle_lib):
    case = small_case(13, dtype="f16", B=5, H=4, Hk=2, D=64, bs=16, lens=(3, 70, 1, 200, 16))
    a, _ = run_oracle(oracle_lib, case, nthreads=1)
    b, _ = run_oracle(oracle_lib, case, nthreads=3)
    np.testing.assert_array_equal(a, b)


# ------------------------------------------------------------- error paths
def test_bad_block_id_and_length_are_flagged(oracle_lib):
    case = small_case(14, dtype="f32", B=3, H=2, Hk=2, D=64, bs=16, lens=(20, 20, 20))
    tables = case["block_tables"].copy()
    NB = case["k_cache"].shape[0]
    tables[1, 1] = NB                       # past the pool
    lens = case["context_lens"].copy()
    lens[2] = tables.shape[1] * 16 + 1      # longer than the table can cover
    c = dict(case, context_lens=lens)
    out, st = run_oracle(oracle_lib, c, tables=tables)
    assert st == (oracle_lib.BAD_BLOCK | oracle_lib.BAD_LEN)
    assert not out[1].any() and not out[2].any()
    good, _ = run_oracle(oracle_lib, case)
    np.testing.assert_array_equal(out[0], good[0])


def test_empty_context_gives_zeros(oracle_lib):
    case = small_case(15, dtype="f32", B=2, H=2, Hk=2, D=64, bs=16, lens=(0, 5))
    out, st = run_oracle(oracle_lib, case)
    assert st == 0 and not out[0].any() and out[1].any()


# ------------------------------------------------------- scatter and copy
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_reshape_and_cache_matches_fancy_index(oracle_lib, dtype):
    g = torch.Generator().manual_seed(21)
    NB, Hk, bs, D, T = 12, 3, 16, 64, 40
    dt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    kc = torch.randn(NB, Hk, bs, D, generator=g).to(dt)
    vc = torch.randn(NB, Hk, bs, D, generator=g).to(dt)
    key = torch.randn(T, Hk, D, generator=g).to(dt)
    val = torch.randn(T, Hk, D, generator=g).to(dt)
    # distinct slots, the pool's first and last among them
    inner = torch.randperm(NB * bs - 2, generator=g)[:T - 2].numpy().astype(np.int64) + 1
    slots = np.concatenate([[0], inner, [NB * bs - 1]]).astype(np.int64)
    slots[3] = -1                                   # padding token: skipped
    k_or, v_or = raw_np(kc).copy(), raw_np(vc).copy()
    st = oracle_lib.reshape_and_cache(raw_np(key), raw_np(val), k_or, v_or, slots)
    assert st == 0
    k_ref, v_ref = raw_np(kc).copy(), raw_np(vc).copy()
    keep = slots >= 0
    b, o = slots[keep] // bs, slots[keep] % bs
    k_ref[b, :, o, :] = raw_np(key)[keep]
    v_ref[b, :, o, :] = raw_np(val)[keep]
    np.testing.assert_array_equal(k_or.view(np.uint8), k_ref.view(np.uint8))
    np.testing.assert_array_equal(v_or.view(np.uint8), v_ref.view(np.uint8))
    bad = slots.copy(); bad[0] = NB * bs
    st = oracle_lib.reshape_and_cache(raw_np(key), raw_np(val), k_or, v_or, bad)
    assert st == oracle_lib.BAD_SLOT


def test_reshape_then_gather_reads_back(oracle_lib):
    """Tokens written through slot = table[pos // bs] * bs + pos % bs come back
    in logical order through the same table."""
    rng = np.random.default_rng(22)
    NB, Hk, bs, D, L = 20, 2, 8, 64, 45
    table = rng.permutation(NB)[: -(-L // bs)].astype(np.int32)
    K = rng.standard_normal((L, Hk, D)).astype(np.float32)
    V = rng.standard_normal((L, Hk, D)).astype(np.float32)
    pos = np.arange(L)
    slots = (table[pos // bs].astype(np.int64) * bs + pos % bs)
    kc = np.zeros((NB, Hk, bs, D), np.float32); vc = np.zeros_like(kc)
    assert oracle_lib.reshape_and_cache(K, V, kc, vc, slots) == 0
    np.testing.assert_array_equal(kc[table[pos // bs], :, pos % bs, :], K)
    np.testing.assert_array_equal(vc[table[pos // bs], :, pos % bs, :], V)


def test_copy_blocks_matches_slices(oracle_lib):
    rng = np.random.default_rng(23)
    layers, NB = 3, 10
    ks = [rng.standard_normal((NB, 2, 16, 64)).astype(np.float32) for _ in range(layers)]
    vs = [rng.standard_normal((NB, 2, 16, 64)).astype(np.float32) for _ in range(layers)]
    ref_k = [k.copy() for k in ks]; ref_v = [v.copy() for v in vs]
    pairs = np.array([[1, 7], [2, 8], [1, 9]], dtype=np.int64)
    assert oracle_lib.copy_blocks(ks, vs, pairs) == 0
    for l in range(layers):
        for s, d in pairs:
            ref_k[l][d] = ref_k[l][s]; ref_v[l][d] = ref_v[l][s]
        np.testing.assert_array_equal(ks[l], ref_k[l])
        np.testing.assert_array_equal(vs[l], ref_v[l])
    assert oracle_lib.copy_blocks(ks, vs, np.array([[0, NB]])) == oracle_lib.BAD_BLOCK


def test_swap_blocks_matches_slices_and_round_trips(oracle_lib):
    """Swap-out copies each pair's gpu block into its host block for every
    layer's K and V (numpy fancy indexing is the definition); swap-in of the
    same pairs after the gpu blocks were overwritten restores them; an id
    outside either pool is skipped and flagged."""
    rng = np.random.default_rng(29)
    layers, NB, NH = 2, 12, 5
    gk = [rng.standard_normal((NB, 2, 16, 64)).astype(np.float32) for _ in range(layers)]
    gv = [rng.standard_normal((NB, 2, 16, 64)).astype(np.float32) for _ in range(layers)]
    hk = [np.zeros((NH, 2, 16, 64), np.float32) for _ in range(layers)]
    hv = [np.zeros((NH, 2, 16, 64), np.float32) for _ in range(layers)]
    pairs = np.array([[3, 0], [11, 4], [5, 2]], dtype=np.int64)
    saved_k = [k.copy() for k in gk]; saved_v = [v.copy() for v in gv]
    assert oracle_lib.swap_blocks(gk, gv, hk, hv, pairs, 0) == 0
    for l in range(layers):
        np.testing.assert_array_equal(hk[l][pairs[:, 1]], gk[l][pairs[:, 0]])
        np.testing.assert_array_equal(hv[l][pairs[:, 1]], gv[l][pairs[:, 0]])
        untouched = np.setdiff1d(np.arange(NH), pairs[:, 1])
        assert not hk[l][untouched].any() and not hv[l][untouched].any()
        gk[l][pairs[:, 0]] = -1.0; gv[l][pairs[:, 0]] = -2.0     # the blocks are reused meanwhile
    assert oracle_lib.swap_blocks(gk, gv, hk, hv, pairs, 1) == 0
    for l in range(layers):
        np.testing.assert_array_equal(gk[l], saved_k[l])
        np.testing.assert_array_equal(gv[l], saved_v[l])
    assert oracle_lib.swap_blocks(gk, gv, hk, hv, np.array([[NB, 0]]), 0) == oracle_lib.BAD_BLOCK
    assert oracle_lib.swap_blocks(gk, gv, hk, hv, np.array([[0, NH]]), 1) == oracle_lib.BAD_BLOCK
    for l in range(layers):
        np.testing.assert_array_equal(gk[l], saved_k[l])


# --------------------------------------------------------- copy-on-write
def test_copy_on_write_rule():
    """Six samples fork a 37-token prompt (partial last block of 16): samples
    0..4 copy the shared partial block on their first write, sample 5 writes in
    place; full prompt blocks stay shared."""
    from oracle.block_manager import OracleBlockManager
    bm = OracleBlockManager(num_blocks=64, block_size=16)
    bm.add_sequence(0, 37)
    prompt = list(bm.tables[0])
    for c in range(1, 6):
        bm.fork(0, c)
    pairs = []
    for s in range(6):
        slot, pair = bm.append_token(s)
        if pair:
            pairs.append(pair)
        assert slot // 16 == bm.tables[s][2] and slot % 16 == 5
    assert len(pairs) == 5 and all(p[0] == prompt[2] for p in pairs)
    assert len({p[1] for p in pairs}) == 5
    assert bm.tables[5][2] == prompt[2]
    for s in range(6):
        assert bm.tables[s][:2] == prompt[:2]
    assert bm.refcount[prompt[0]] == 6 and bm.refcount[prompt[2]] == 1
    # A block-aligned prompt has no partial block: every sample takes a fresh block.
    bm2 = OracleBlockManager(num_blocks=64, block_size=16)
    bm2.add_sequence(0, 32)
    for c in range(1, 6):
        bm2.fork(0, c)
    assert all(bm2.append_token(s)[1] is None for s in range(6))


# ---------------------------------------------------------- prefix caching
# The page "PagedAttention: Efficient LLM Serving with vLLM", "Advanced
# Features": Prefix Caching (the first request with a prefix computes its KV
# blocks and caches them; later requests with the same prefix reuse them) and
# KV-Cache Sharing (only the divergent tokens get new blocks).  Every count
# below is worked out by hand from those statements and the block-count rule
# (100 tokens at 16 per block: 6 full blocks + 4 tokens in a 7th).

def _prompt(n, seed):
    return [int(x) for x in np.random.default_rng(seed).integers(0, 32000, n)]


def test_prefix_cache_first_request_computes_later_ones_reuse():
    from oracle.block_manager import OraclePrefixCache
    bs, system = 16, _prompt(100, 1)
    pc = OraclePrefixCache(num_blocks=64, block_size=bs)
    reqs = [system + _prompt(20, 10 + i) for i in range(5)]       # 120 tokens: 8 blocks each
    first, cached = pc.allocate_prompt(reqs[0])
    assert cached == 0 and len(first) == 8 and len(set(first)) == 8
    pc.commit_prompt(reqs[0], first)
    tables = [first]
    for r in reqs[1:]:
        t, cached = pc.allocate_prompt(r)
        assert cached == 96                        # the 6 full system-prompt blocks
        assert t[:6] == first[:6]                  # reused, not recomputed
        assert len(t) == 8 and not set(t[6:]) & set(b for u in tables for b in u)
        pc.commit_prompt(r, t)
        tables.append(t)
    assert all(pc.holders[b] == 5 for b in first[:6])
    assert all(pc.holders[b] == 1 for t in tables for b in t[6:])
    # 6 shared + 5 x 2 own blocks, against 5 x 8 without the cache
    assert len({b for t in tables for b in t}) == 16
    assert pc.available() == 64 - 16
    # two requests for a new prompt that arrive before either is committed
    # both compute it; the first commit's blocks are the ones later reused
    other = _prompt(48, 2)
    a, _ = pc.allocate_prompt(other)
    b, _ = pc.allocate_prompt(other)
    pc.commit_prompt(other, a)
    pc.commit_prompt(other, b)
    c, cached = pc.allocate_prompt(other + [7])
    assert cached == 48 and c[:3] == a[:3] and not set(c[:3]) & set(b)


def test_prefix_cache_key_covers_every_earlier_token():
    from oracle.block_manager import OraclePrefixCache
    bs, p = 16, _prompt(64, 3)
    pc = OraclePrefixCache(num_blocks=32, block_size=bs)
    t, _ = pc.allocate_prompt(p)
    pc.commit_prompt(p, t)
    # blocks 1..3 hold the same tokens after a different block 0: no reuse
    q = list(p)
    q[3] += 1
    u, cached = pc.allocate_prompt(q)
    assert cached == 0 and not set(u) & set(t)
    # the same first 40 tokens: the 2 full blocks they cover
    v, cached = pc.allocate_prompt(p[:40] + _prompt(30, 4))
    assert cached == 32 and v[:2] == t[:2] and v[2] not in t
    # block 0 of another committed prompt, then block 1 of p: block 0 is
    # reused, block 1 is not (its K/V in p was computed after p's block 0)
    x = _prompt(32, 7)
    tx, _ = pc.allocate_prompt(x)
    pc.commit_prompt(x, tx)
    mixed = x[:16] + p[16:32]
    w, cached = pc.allocate_prompt(mixed)
    assert cached == 16 and w[0] == tx[0] and w[1] not in t and w[1] != tx[1]


def test_only_divergent_tokens_get_new_blocks():
    """Six samples of one 100-token prompt: they share its 7 blocks; each
    sample's first new token copies the shared partial block (samples 0-4;
    sample 5 is its last holder and writes in place); 20 tokens later every
    sample holds one more block of its own."""
    from oracle.block_manager import OraclePrefixCache
    bs = 16
    pc = OraclePrefixCache(num_blocks=64, block_size=bs)
    prompt, _ = pc.allocate_prompt(_prompt(100, 5))
    tables = [list(prompt)]
    for _ in range(5):
        pc.fork(prompt)
        tables.append(list(prompt))
    pairs = []
    for s in range(6):
        slot, pair = pc.append_token(tables[s], 100)
        assert slot == tables[s][6] * bs + 4
        if pair:
            pairs.append(pair)
    assert len(pairs) == 5 and all(p[0] == prompt[6] for p in pairs)
    assert tables[5][6] == prompt[6]
    for n in range(101, 120):
        for s in range(6):
            assert pc.append_token(tables[s], n)[1] is None
    assert all(t[:6] == prompt[:6] for t in tables)
    assert all(pc.holders[b] == 6 for b in prompt[:6])
    # 6 shared + 6 partial-block copies (5 copies + the original) + 6 new
    assert len({b for t in tables for b in t}) == 18
    assert all(len(t) == 8 for t in tables)


def test_cached_block_is_copied_before_a_write():
    """A committed block is read by every later request that reuses it, so
    its only holder writes into a copy; the entry stays reusable."""
    from oracle.block_manager import OraclePrefixCache
    bs, p = 8, _prompt(24, 6)
    pc = OraclePrefixCache(num_blocks=16, block_size=bs)
    t, _ = pc.allocate_prompt(p)
    pc.commit_prompt(p, t)
    old = t[2]
    assert pc.prepare_write(t, 2) == (old, t[2]) and t[2] != old
    assert pc.holders[old] == 0 and pc.is_cached(old)
    assert pc.prepare_write(t, 2) is None                  # the copy is private
    again, cached = pc.allocate_prompt(p)
    assert cached == 24 and again == [t[0], t[1], old]


def test_released_prefix_stays_reusable_and_the_longest_released_goes_first():
    """The eviction rule: a cached block nobody holds keeps its entry until a
    block is needed and none is free; then the one released longest ago."""
    from oracle.block_manager import OraclePrefixCache
    bs, NB = 8, 12
    pc = OraclePrefixCache(num_blocks=NB, block_size=bs)
    p1, p2 = list(range(16)), list(range(100, 116))
    t1, _ = pc.allocate_prompt(p1)
    pc.commit_prompt(p1, t1)
    t2, _ = pc.allocate_prompt(p2)
    pc.commit_prompt(p2, t2)
    assert (t1, t2) == ([0, 1], [2, 3])                   # block 0 first
    pc.release(t1)                                        # released first
    pc.release(t2)
    assert pc.available() == NB and pc.idle == [0, 1, 2, 3]
    again, cached = pc.allocate_prompt(p1)                # still reusable
    assert cached == 16 and again == t1
    pc.release(again)                                     # p1 is now the latest released
    assert pc.idle == [2, 3, 0, 1]
    assert sorted(pc.allocate(8)) == list(range(4, 12))   # the free blocks go first
    assert pc.allocate(2) == [2, 3]                       # then p2's: released longest ago
    assert not pc.is_cached(2) and not pc.is_cached(3)
    _, cached = pc.allocate_prompt(p2)
    assert cached == 0
    pc2 = OraclePrefixCache(num_blocks=NB, block_size=bs)
    u1, _ = pc2.allocate_prompt(p1)
    pc2.commit_prompt(p1, u1)
    pc2.release(u1)
    pc2.allocate(NB - 2)
    _, cached = pc2.allocate_prompt(p1)                   # p1 survived
    assert cached == 16


def test_refused_request_changes_nothing():
    """A request that cannot get every block it needs takes none and leaves
    the pool as it was: a reused block nobody holds cannot also serve as
    one of the request's fresh blocks."""
    from oracle.block_manager import OraclePrefixCache
    bs = 8
    pc = OraclePrefixCache(num_blocks=4, block_size=bs)
    p = list(range(16))
    t, _ = pc.allocate_prompt(p)
    pc.commit_prompt(p, t)
    pc.release(t)                                   # 2 idle cached + 2 free
    keep = pc.allocate(1)                           # 2 idle + 1 free
    state = (list(pc.free), list(pc.idle), list(pc.holders))
    assert pc.allocate_prompt(p + list(range(50, 66))) is None   # 2 reused + 2 fresh > 1 free
    assert (list(pc.free), list(pc.idle), list(pc.holders)) == state
    t3, cached = pc.allocate_prompt(p + [1, 2])     # 2 reused + 1 fresh: fits
    assert cached == 16 and t3[:2] == t and t3[2] not in keep
