"""The host block pool with prefix caching (pkv_block_pool_*), on the CPU.

Without prefix caching the pool must hand out exactly the blocks the
oracle's block manager does (on-demand allocation, forks, copy-on-write and
frees on the page "PagedAttention: Efficient LLM Serving with vLLM", "The
PagedAttention Algorithm" and "Advanced Features"); with it, exactly the
blocks of the oracle's prefix-cache model: a request whose prompt starts with
the tokens of committed full blocks reuses those blocks ("Advanced
Features", Prefix Caching)."""
import os

import numpy as np
import pytest

import paged_kv_cache_311_gb300 as pkv
from oracle.block_manager import OracleBlockManager, OraclePrefixCache
from paged_kv_cache_311_gb300.build import build, library_path
from tests.util import read_golden


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not os.path.exists(library_path()):
        build()
    return pkv.load_library()


def test_blocks_on_demand_worked_example():
    _, rows = read_golden("worked_example_blocks.txt")
    for tokens, bs, blocks, slots, unused in rows:
        pool = pkv.BlockPool(64, bs)
        table, cached = pool.allocate_prompt(np.arange(tokens))
        assert (len(table), cached) == (blocks, 0)
        np.testing.assert_array_equal(table, np.arange(blocks))    # block 0 first
        assert pool.available() == 64 - blocks


def test_same_blocks_as_the_oracle_block_manager_without_caching():
    """Random adds, token appends (a new block when the last is full, a
    copy when it is shared), forks and frees: tables, copy pairs and
    refcounts follow the oracle's block manager step for step."""
    rng = np.random.default_rng(8)
    bs, NB = 16, 400
    pool, ref = pkv.BlockPool(NB, bs), OracleBlockManager(NB, bs)
    tables, lens, nxt = {}, {}, 0
    for step in range(600):
        op = rng.random()
        live = sorted(tables)
        if op < 0.15 or not live:
            n = int(rng.integers(1, 70))
            if pool.available() < -(-n // bs) + 8:
                continue
            tb, cached = pool.allocate_prompt(rng.integers(0, 1000, n))
            assert cached == 0
            assert list(tb) == ref.add_sequence(nxt, n)
            tables[nxt], lens[nxt] = tb, n
            nxt += 1
        elif op < 0.25:
            s = int(rng.choice(live))
            pool.fork(tables[s])
            ref.fork(s, nxt)
            tables[nxt], lens[nxt] = tables[s].copy(), lens[s]
            nxt += 1
        elif op < 0.35:
            s = int(rng.choice(live))
            pool.release(tables.pop(s))
            lens.pop(s)
            ref.free_sequence(s)
        else:
            s = int(rng.choice(live))
            if pool.available() < 2:
                continue
            slot, ref_pair = ref.append_token(s)
            j, off = divmod(lens[s], bs)
            if off == 0:
                tables[s] = np.append(tables[s], pool.allocate(1)).astype(np.int32)
                pair = None
            else:
                pair = pool.prepare_write(tables[s], j)
            lens[s] += 1
            assert pair == ref_pair
            assert tables[s][j] * bs + off == slot
        for s in tables:
            assert list(tables[s]) == ref.tables[s]
    for b in range(NB):
        assert pool.refcount(b) == ref.refcount[b]
    assert pool.available() == len(ref.free)


def test_prefix_reuse_is_exact_and_chained():
    bs = 16
    pool = pkv.BlockPool(64, bs)
    rng = np.random.default_rng(2)
    sys_prompt = rng.integers(0, 32000, 3 * bs + 5)          # 3 full blocks + 5 tokens
    a = np.concatenate([sys_prompt, rng.integers(0, 32000, 20)])
    ta, ca = pool.allocate_prompt(a)
    assert ca == 0
    pool.commit_prompt(a, ta)
    assert all(pool.is_cached(b) for b in ta[:len(a) // bs]) and not pool.is_cached(ta[-1])
    # same system prompt, another question: its 3 full blocks are reused;
    # block 4 of a held the prompt's 5 last tokens plus a's own: no match
    b = np.concatenate([sys_prompt, rng.integers(0, 32000, 30)])
    tb, cb = pool.allocate_prompt(b)
    assert cb == 3 * bs
    np.testing.assert_array_equal(tb[:3], ta[:3])
    assert len(set(tb[3:]) & set(ta)) == 0
    assert [pool.refcount(x) for x in ta[:3]] == [2, 2, 2]
    # the same tokens for block 2 after a different block 1: only block 0 matches
    c = a.copy()
    c[bs + 3] += 1
    tc, cc = pool.allocate_prompt(c)
    assert cc == bs and tc[0] == ta[0] and tc[2] != ta[2]
    # a prompt ending inside a cached block reuses only the full blocks before
    td, cd = pool.allocate_prompt(a[:2 * bs + 7])
    assert cd == 2 * bs and list(td[:2]) == list(ta[:2]) and td[2] != ta[2]
    st = pool.stats()
    assert st["hits"] == 3 + 1 + 2


def test_released_prefix_stays_cached_until_evicted_least_recent_first():
    bs, NB = 8, 12
    pool = pkv.BlockPool(NB, bs)
    p1, p2 = np.arange(2 * bs), np.arange(100, 100 + 2 * bs)
    t1, _ = pool.allocate_prompt(p1); pool.commit_prompt(p1, t1)
    t2, _ = pool.allocate_prompt(p2); pool.commit_prompt(p2, t2)
    pool.release(t1)                      # released first: evicted first
    pool.release(t2)
    assert pool.available() == NB
    assert pool.stats()["evictable"] == 4
    again, cached = pool.allocate_prompt(p1)   # still reusable
    assert cached == 2 * bs and list(again) == list(t1)
    pool.release(again)                   # now p1 is the most recently released
    filler = pool.allocate(8)              # the 8 free blocks
    assert not set(filler) & set(t1) | set(filler) & set(t2)
    more = pool.allocate(2)                # evicts p2's blocks (least recently released)
    assert set(more) == set(t2)
    _, c2 = pool.allocate_prompt(p1)       # p1 survived
    assert c2 == 2 * bs


def test_out_of_blocks_takes_nothing():
    pool = pkv.BlockPool(6, 16)
    t, _ = pool.allocate_prompt(np.arange(70))          # 5 blocks
    pool.commit_prompt(np.arange(70), t)
    with pytest.raises(pkv.PkvError):
        pool.allocate_prompt(np.concatenate([np.arange(64), np.arange(900, 950)]))  # 4 reused + 4 new
    assert pool.available() == 1
    assert [pool.refcount(b) for b in t] == [1] * 5
    with pytest.raises(pkv.PkvError):
        pool.allocate(2)
    assert pool.available() == 1


def test_writing_into_a_cached_block_copies_it():
    """A cached block is shared with every later request that reuses it, so
    a write into it (its sole holder included) goes to a copy."""
    bs = 8
    pool = pkv.BlockPool(16, bs)
    p = np.arange(3 * bs)
    t, _ = pool.allocate_prompt(p)
    pool.commit_prompt(p, t)
    pair = pool.prepare_write(t, 2)
    assert pair is not None and pair[0] == 2 and t[2] == pair[1]
    assert pool.refcount(2) == 0 and pool.is_cached(2)   # the entry stays reusable
    assert pool.prepare_write(t, 2) is None               # the copy is private


def test_prefix_cache_follows_the_oracle_model():
    """A random walk of prompts over five shared prefixes (some committed,
    some not), releases and refused requests: the pool hands out the tables
    and cached-token counts of the oracle's prefix-cache model, and holder
    counts, cache entries and the free count agree throughout.  The model is
    pinned to the page's prefix-caching statements in the oracle pins."""
    rng = np.random.default_rng(21)
    bs, NB = 8, 60
    pool, model = pkv.BlockPool(NB, bs), OraclePrefixCache(NB, bs)
    prefixes = [rng.integers(0, 50, int(rng.integers(4, 40))) for _ in range(5)]
    live = []
    refused = 0
    for step in range(800):
        if live and (rng.random() < 0.4 or model.available() < 2):
            i = int(rng.integers(0, len(live)))
            toks, table = live.pop(i)
            pool.release(table)
            model.release(list(table))
        else:
            pre = prefixes[int(rng.integers(0, len(prefixes)))]
            toks = np.concatenate([pre[:int(rng.integers(0, len(pre) + 1))],
                                   rng.integers(0, 50, int(rng.integers(0, 20)))]).astype(np.int32)
            if toks.size == 0:
                continue
            want = model.allocate_prompt(toks.tolist())
            if want is None:
                refused += 1
                with pytest.raises(pkv.PkvError):
                    pool.allocate_prompt(toks)
                continue
            table, cached = pool.allocate_prompt(toks)
            assert (list(table), cached) == (want[0], want[1])
            if rng.random() < 0.8:
                pool.commit_prompt(toks, table)
                model.commit_prompt(toks.tolist(), list(table))
            live.append((toks, table))
        assert pool.available() == model.available()
    for b in range(NB):
        assert pool.refcount(b) == model.holders[b]
        assert pool.is_cached(b) == model.is_cached(b)
    st = pool.stats()
    assert (st["lookups"], st["hits"]) == (model.lookups, model.hits)
    assert st["hits"] > 100          # the walk reused cached prefixes often
    assert refused > 0               # and ran into a full pool


def test_refused_prompt_leaves_the_eviction_order_alone():
    """A refused request takes nothing and leaves the order in which idle
    cached blocks are evicted as it was."""
    bs = 8
    pool, model = pkv.BlockPool(6, bs), OraclePrefixCache(6, bs)
    p1, p2 = np.arange(16, dtype=np.int32), np.arange(100, 116, dtype=np.int32)
    for p in (p1, p2):
        t, _ = pool.allocate_prompt(p); pool.commit_prompt(p, t)
        u = model.allocate_prompt(p.tolist())[0]; model.commit_prompt(p.tolist(), u)
        pool.release(t); model.release(u)
    assert list(pool.allocate(1)) == model.allocate(1) == [4]
    # p1 + 4 more blocks: 2 reused (idle) + 4 fresh, but only 1 free + 2 other idle blocks
    big = np.concatenate([p1, np.arange(500, 532, dtype=np.int32)])
    assert model.allocate_prompt(big.tolist()) is None
    with pytest.raises(pkv.PkvError):
        pool.allocate_prompt(big)
    # the free block, then p1's blocks: still the ones released longest ago
    assert list(pool.allocate(3)) == model.allocate(3) == [5, 0, 1]
    assert not pool.is_cached(0) and pool.is_cached(2)


def test_system_prompt_requests_share_cached_blocks_and_group():
    """Requests for 3 system prompts arrive interleaved; each prompt's first
    request computes and commits it, every later one reuses its full blocks
    (cached_tokens = those blocks' tokens).  The planner then groups each
    prompt's requests across their batch positions."""
    bs, G = 16, 4
    rng = np.random.default_rng(12)
    prompts = [rng.integers(0, 32000, int(n)) for n in (200, 333, 128)]
    pool = pkv.BlockPool(400, bs)
    tables, lens, which = [], [], []
    for i in range(18):
        p = i % 3
        toks = np.concatenate([prompts[p], rng.integers(0, 32000, int(rng.integers(5, 40)))])
        t, cached = pool.allocate_prompt(toks)
        assert cached == (0 if i < 3 else len(prompts[p]) // bs * bs)
        pool.commit_prompt(toks, t)
        tables.append(t); lens.append(len(toks)); which.append(p)
    for p in range(3):
        full = len(prompts[p]) // bs
        first = tables[p][:full]
        for i in range(p, 18, 3):
            np.testing.assert_array_equal(tables[i][:full], first)
            assert pool.refcount(int(first[0])) == 6
    MB = max(len(t) for t in tables)
    bt = np.full((18, MB), -1, np.int32)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = t
    from tests.test_planner import check_coverage
    plan = pkv.plan_shared_prefix(bt, np.array(lens, np.int32), 16, 4, 128, bs, max(lens), 256)
    items, _ = check_coverage(plan, bt, np.array(lens, np.int32), G, 4)
    groups = {frozenset(it[7]) for it in items if it[1] > G}
    assert groups == {frozenset(range(p, 18, 3)) for p in range(3)}


def _per_sequence_append(pool, tables, lens):
    """One call per sequence, in batch order: the reference for append_slots."""
    bs = pool.block_size
    slots, pairs = [], []
    for s in range(len(tables)):
        j, off = divmod(int(lens[s]), bs)
        if off == 0:
            tables[s] = np.append(tables[s], pool.allocate(1)).astype(np.int32)
        else:
            pair = pool.prepare_write(tables[s], j)
            if pair:
                pairs.append(pair)
        slots.append(int(tables[s][j]) * bs + off)
    return slots, pairs


def test_append_slots_equals_one_call_per_sequence():
    """Random histories (prompts reusing cached prefixes, forks, releases)
    kept in two pools: one steps its batch with append_slots, the other with
    a call per sequence. Tables, slots, copy pairs, holders and the free
    count agree at every step."""
    rng = np.random.default_rng(31)
    bs, NB, MB = 8, 300, 64
    a, b = pkv.BlockPool(NB, bs), pkv.BlockPool(NB, bs)
    prefixes = [rng.integers(0, 40, int(rng.integers(8, 60))).astype(np.int32) for _ in range(3)]
    seqs = []   # (table for pool a as a padded row, table for pool b, length)
    for step in range(150):
        op = rng.random()
        if op < 0.25 or not seqs:
            pre = prefixes[int(rng.integers(0, 3))]
            toks = np.concatenate([pre, rng.integers(0, 40, int(rng.integers(0, 12)))]).astype(np.int32)
            if a.available() < toks.size // bs + 4:
                continue
            ta, _ = a.allocate_prompt(toks)
            tb, _ = b.allocate_prompt(toks)
            assert np.array_equal(ta, tb)
            if rng.random() < 0.7:
                a.commit_prompt(toks, ta)
                b.commit_prompt(toks, tb)
            seqs.append([ta, tb, toks.size])
        elif op < 0.35:
            k = int(rng.integers(0, len(seqs)))
            a.fork(seqs[k][0])
            b.fork(seqs[k][1])
            seqs.append([seqs[k][0].copy(), seqs[k][1].copy(), seqs[k][2]])
        elif op < 0.45:
            k = int(rng.integers(0, len(seqs)))
            ta, tb, _ = seqs.pop(k)
            a.release(ta)
            b.release(tb)
        else:
            live = [s for s in seqs if s[2] // bs < MB]
            if not live or a.available() < len(live):
                continue
            rows = np.full((len(live), MB), -1, np.int32)
            for i, s in enumerate(live):
                rows[i, :s[0].size] = s[0]
            lens = np.array([s[2] for s in live], np.int32)
            slots, pairs = a.append_slots(rows, lens)
            tabs_b = [s[1] for s in live]
            want_slots, want_pairs = _per_sequence_append(b, tabs_b, lens)
            assert slots.tolist() == want_slots
            assert [tuple(p) for p in pairs.tolist()] == want_pairs
            for i, s in enumerate(live):
                n = -(-(int(lens[i]) + 1) // bs)
                s[0] = rows[i, :n].copy()
                s[1] = tabs_b[i]
                s[2] += 1
                assert np.array_equal(s[0], s[1])
        assert a.available() == b.available()
    for blk in range(NB):
        assert a.refcount(blk) == b.refcount(blk) and a.is_cached(blk) == b.is_cached(blk)


def test_append_slots_copy_on_write_rule_in_one_call():
    """Six samples forked from a 37-token prompt, stepped in one call: samples
    0-4 copy the shared partial block, sample 5 writes in place, and every
    slot is offset 5 of the sample's third block ("Advanced Features",
    KV-Cache Sharing)."""
    bs = 16
    pool = pkv.BlockPool(64, bs)
    t0 = pool.allocate(3)
    for _ in range(5):
        pool.fork(t0)
    rows = np.tile(np.append(t0, [-1, -1]).astype(np.int32), (6, 1))
    slots, pairs = pool.append_slots(rows, np.full(6, 37, np.int32))
    assert pairs.shape == (5, 2) and (pairs[:, 0] == t0[2]).all()
    assert len(set(pairs[:, 1].tolist())) == 5
    assert rows[5, 2] == t0[2] and all(rows[s, 2] != t0[2] for s in range(5))
    assert (slots == rows[:, 2].astype(np.int64) * bs + 5).all()
    assert (rows[:, :2] == t0[:2]).all() and pool.refcount(int(t0[0])) == 6


def test_append_slots_stops_where_the_pool_runs_out():
    bs = 8
    pool = pkv.BlockPool(5, bs)
    t = pool.allocate(4)                       # four one-block sequences, each full
    rows = np.full((4, 4), -1, np.int32)
    rows[:, 0] = t
    before = rows.copy()
    with pytest.raises(pkv.PkvError) as e:
        pool.append_slots(rows, np.full(4, bs, np.int32))   # each needs a new block; 1 is left
    assert e.value.status == -4 and e.value.done == 1
    assert rows[0, 1] >= 0 and (rows[1:] == before[1:]).all()
    assert pool.available() == 0


def test_append_slots_checks_every_row_first():
    bs = 8
    pool = pkv.BlockPool(16, bs)
    t = pool.allocate(2)
    rows = np.array([[t[0], -1], [t[1], -1]], np.int32)
    # a negative length; no room for block index 2; a block nobody holds
    for lens in ([3, -1], [3, 16], [8, 5]):
        r = rows.copy()
        if lens == [8, 5]:
            r[1, 0] = 15                           # a block nobody holds
        with pytest.raises(pkv.PkvError) as e:
            pool.append_slots(r, np.array(lens, np.int32))
        assert e.value.status == -1
        assert pool.available() == 14


def test_append_slots_follows_the_oracle_block_manager():
    """Random adds, forks and frees; at each decode step every live sequence
    gets its next token through one append_slots call, and the oracle's block
    manager takes the same tokens one sequence at a time in batch order:
    slots, copy pairs, tables and holder counts agree."""
    rng = np.random.default_rng(47)
    bs, NB, MB = 16, 500, 40
    pool, ref = pkv.BlockPool(NB, bs), OracleBlockManager(NB, bs)
    tables, lens, nxt = {}, {}, 0
    for step in range(300):
        op = rng.random()
        live = sorted(tables)
        if op < 0.15 or not live:
            n = int(rng.integers(1, 120))
            if pool.available() < -(-n // bs) + 40:
                continue
            tb, _ = pool.allocate_prompt(rng.integers(0, 1000, n))
            assert list(tb) == ref.add_sequence(nxt, n)
            tables[nxt], lens[nxt] = tb, n
            nxt += 1
        elif op < 0.3:
            s = int(rng.choice(live))
            pool.fork(tables[s])
            ref.fork(s, nxt)
            tables[nxt], lens[nxt] = tables[s].copy(), lens[s]
            nxt += 1
        elif op < 0.4:
            s = int(rng.choice(live))
            pool.release(tables.pop(s))
            lens.pop(s)
            ref.free_sequence(s)
        else:
            batch = [s for s in live if lens[s] // bs < MB]
            if not batch or pool.available() < len(batch):
                continue
            rows = np.full((len(batch), MB), -1, np.int32)
            for i, s in enumerate(batch):
                rows[i, :tables[s].size] = tables[s]
            slots, pairs = pool.append_slots(rows, np.array([lens[s] for s in batch], np.int32))
            want_pairs = []
            for i, s in enumerate(batch):
                slot, pair = ref.append_token(s)
                assert slots[i] == slot
                if pair:
                    want_pairs.append(pair)
                lens[s] += 1
                tables[s] = rows[i, :-(-lens[s] // bs)].copy()
                assert list(tables[s]) == ref.tables[s]
            assert [tuple(p) for p in pairs.tolist()] == want_pairs
    for b in range(NB):
        assert pool.refcount(b) == ref.refcount[b]
    assert pool.available() == len(ref.free)


def test_decode_batch_system_prompt_follows_the_oracle_model():
    """DecodeBatch on the pool: 40 requests over 3 system prompts, then 20
    decode steps; every table, cached count, slot and copy pair matches the
    oracle's prefix-cache model."""
    from tests.pool_lockstep import Lockstep, build_system_prompt, system_prompt_requests
    bs = 16
    reqs, prompts = system_prompt_requests(5, 40, 3, (100, 300), (1, 40))
    ls = Lockstep(600, bs, 40, 32)
    pre = build_system_prompt(ls, reqs)
    # the first request of each prompt computes it; later ones reuse its full blocks
    assert [c for _, c in pre] == [0, 0, 0] + [len(prompts[i % 3]) // bs * bs for i in range(3, 40)]
    assert [s.size for s, _ in pre] == [len(r) - c for r, (_, c) in zip(reqs, pre)]
    for _ in range(20):
        ls.step(40)
    ls.check_holders()


def test_decode_batch_sampling_follows_the_oracle_model():
    """Eight prompts forked into six samples each, then 20 steps: the first
    step copies every shared partial last block (five copies per prompt whose
    length is not a multiple of the block size), as the oracle model does."""
    from tests.pool_lockstep import Lockstep, build_sampling, sampling_prompts
    bs, S = 16, 6
    prompts = sampling_prompts(6, 8, (40, 200))
    ls = Lockstep(400, bs, 8 * S, 32)
    build_sampling(ls, prompts, S)
    _, pairs = ls.step(8 * S)
    assert pairs.shape[0] == 5 * sum(1 for p in prompts if p.size % bs)
    for _ in range(19):
        ls.step(8 * S)
    ls.check_holders()
