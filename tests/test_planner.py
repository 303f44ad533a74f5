"""The host planner of the shared-prefix decode (pkv_plan_shared_prefix), on
the CPU: the plan must cover every token of every sequence exactly once for
each of its query rows, only group sequences that really share leading
blocks, and size the workspace for the partials it creates."""
import numpy as np
import pytest

import paged_kv_cache_311_gb300 as pkv
from paged_kv_cache_311_gb300.build import build, library_path
from workloads import PagedDecodeWorkload, get


@pytest.fixture(scope="module", autouse=True)
def lib():
    import os
    if not os.path.exists(library_path()):
        build()
    return pkv.load_library()


def decode_plan(plan, B, Hk, G):
    h = plan.host
    n_items, slots, nseq, nkv, iints, maxseg = (int(x) for x in h[:6])
    assert (nseq, nkv) == (B, Hk)
    expected = h[8:8 + B]
    items = []
    base = 8 + 2 * B
    for i in range(n_items):
        it = h[base + i * iints: base + (i + 1) * iints]
        seq0, nrows, slot, nseg, tiles, nids, checks = (int(x) for x in it[:7])
        members = [int(x) for x in it[8:8 + nrows // G]]
        assert members[0] == seq0 and all(x == -1 for x in it[8 + nrows // G:32])
        raw = [[int(x) for x in it[32 + 8 * k: 40 + 8 * k]] for k in range(nseg)]
        segs = [tuple(r[:5]) for r in raw]
        ids = it[32 + 8 * maxseg:]
        items.append((seq0, nrows, slot, segs, ids, (tiles, nids, checks), raw, members))
    return items, expected, slots


def check_coverage(plan, tables, lens, G, Hk, bs=16):
    B = len(lens)
    items, expected, slots = decode_plan(plan, B, Hk, G)
    np.testing.assert_array_equal(plan.host[8 + B:8 + 2 * B], lens)   # the lengths it was made for
    covered = [np.zeros(max(int(L), 0), dtype=int) for L in lens]
    slots_seen = [set() for _ in range(B)]
    for seq0, nrows, slot, segs, ids, totals, raw, members in items:
        assert len(set(members)) == len(members)
        assert nrows % G == 0 and nrows <= 24
        if not segs:
            assert lens[seq0] <= 0
            continue
        # the per-segment offsets the kernel reads: 16-token tiles, block ids
        # and device-table checks (every member's table for a shared prefix
        # segment), in segment order, and the item's totals
        t = n = c = 0
        for tseq, tb, te, rlo, rhi, first_tile, id_off, check_off in raw:
            assert (first_tile, id_off, check_off) == (t, n, c)
            nb = -(-te // bs) - tb // bs
            shared = rlo == 0 and rhi == nrows and nrows > G
            t += -(-(te - tb) // 16)
            n += nb
            c += (nrows // G if shared else 1) * nb
        assert totals == (t, n, c)
        # the item carries its segments' physical block ids, in segment order
        want = np.concatenate([tables[tseq][tb // bs: -(-te // bs)] for tseq, tb, te, _, _ in segs])
        assert want.size <= ids.size
        np.testing.assert_array_equal(ids[:want.size], want)
        for tseq, tb, te, rlo, rhi in segs:
            assert rlo % G == 0 and rhi % G == 0
            for m in range(rlo // G, rhi // G):
                s = members[m]
                assert 0 <= tb < te <= lens[s]
                # the tokens come from table_seq's blocks: they must be s's blocks too
                j = np.arange(tb // bs, -(-te // bs))
                np.testing.assert_array_equal(tables[tseq][j], tables[s][j])
                covered[s][tb:te] += 1
                slots_seen[s].add(slot)
    for s in range(B):
        if lens[s] > 0:
            assert (covered[s] == 1).all(), f"sequence {s} not covered exactly once"
            assert slots_seen[s] == set(range(int(expected[s])))
        else:
            assert expected[s] == 0
    assert slots == max(1, int(expected.max()))
    return items, expected


def test_forked_prompts_share_their_full_blocks():
    cfg = get("shared_prefix_bf16")
    w = PagedDecodeWorkload(cfg, 31103, total_steps=2)
    inp = w.next_step()
    plan = pkv.plan_shared_prefix(inp.block_tables, inp.context_lens, cfg.num_heads, cfg.num_kv_heads,
                                  cfg.head_dim, cfg.block_size, inp.max_context_len)
    items, expected = check_coverage(plan, inp.block_tables, inp.context_lens, cfg.group,
                                     cfg.num_kv_heads)
    # every group of 6 samples forms one group (24 rows) whose prefix items
    # read the prompt's full blocks once
    prefix_items = [it for it in items if it[1] == 24]
    for p, lp in enumerate(w.prompt_lens):
        shared = (int(lp) // 16 * 16) // 32 * 32
        mine = [it for it in prefix_items if set(it[7]) == set(range(6 * p, 6 * p + 6))]
        assert sum(seg[2] - seg[1] for it in mine for seg in it[3] if seg[3] == 0 and seg[4] == 24) == shared
    # the items come heaviest first (tokens streamed)
    weights = [sum(s[2] - s[1] for s in it[3]) for it in items]
    assert all(a >= b for a, b in zip(weights, weights[1:]))


def test_automatic_plan_is_one_balanced_wave():
    """partition_size 0: the smallest target T whose items fit one CTA per
    resident slot (3 per SM; 152 SMs when no GPU answers) over the kv heads;
    every item then streams at most T tokens (plus one alignment step)."""
    cfg = get("shared_prefix_bf16")
    w = PagedDecodeWorkload(cfg, 31103, total_steps=8)
    for _ in range(6):
        inp = w.next_step()
    plan = pkv.plan_shared_prefix(inp.block_tables, inp.context_lens, cfg.num_heads, cfg.num_kv_heads,
                                  cfg.head_dim, cfg.block_size, inp.max_context_len)
    items, _ = check_coverage(plan, inp.block_tables, inp.context_lens, cfg.group, cfg.num_kv_heads)
    T = int(plan.host[6])
    tokens = [sum(s[2] - s[1] for s in it[3]) for it in items]
    assert max(tokens) <= T + 32
    assert len(items) * cfg.num_kv_heads <= 3 * 152
    # one step below T would not fit: T is the smallest that does
    smaller = pkv.plan_shared_prefix(inp.block_tables, inp.context_lens, cfg.num_heads,
                                     cfg.num_kv_heads, cfg.head_dim, cfg.block_size,
                                     inp.max_context_len, T - 32)
    assert int(smaller.host[0]) * cfg.num_kv_heads > 3 * 152


def test_no_sharing_gives_plain_partitions():
    cfg = get("llama7b_f16")
    inp = PagedDecodeWorkload(cfg, 1, total_steps=1).next_step()
    plan = pkv.plan_shared_prefix(inp.block_tables, inp.context_lens, 32, 32, 128, 16,
                                  inp.max_context_len, 512)
    items, expected = check_coverage(plan, inp.block_tables, inp.context_lens, 1, 32)
    assert all(it[1] == 1 and len(it[3]) == 1 for it in items)
    np.testing.assert_array_equal(expected, -(-inp.context_lens // 512))


def test_groups_are_cut_at_24_rows_and_long_tails_split():
    bs, G = 16, 4
    prompt = 200
    lens, rows = [], []
    nb_prompt = -(-prompt // bs)
    next_block = nb_prompt
    for m in range(8):                       # 8 forks of one prompt: groups of 6 + 2
        tail = 700 if m == 1 else 5          # one long tail (> partition) is split off
        L = prompt + tail
        own = list(range(next_block, next_block + -(-L // bs) - nb_prompt + 1))
        next_block += len(own)
        rows.append(list(range(nb_prompt - 1)) + own)   # the partial prompt block is copied
        lens.append(L)
    MB = max(len(r) for r in rows)
    bt = np.full((8, MB), -1, np.int32)
    for i, r in enumerate(rows):
        bt[i, :len(r)] = r[:MB]
    lens = np.array(lens, np.int32)
    plan = pkv.plan_shared_prefix(bt, lens, 16, 4, 128, bs, int(lens.max()), 256)
    items, expected = check_coverage(plan, bt, lens, G, 4)
    groups = sorted({(min(it[7]), it[1]) for it in items if it[1] > G})
    assert groups == [(0, 24), (6, 8)]
    # 192 shared tokens plus five folded 13-token tails (a 16-row load each)
    # exceed one 256-token item: the group takes two; the long tail three more
    assert expected[1] == 2 + 3


def test_empty_context_gets_a_zero_item_and_plan_size_is_bounded():
    bt = np.array([[0, 1, -1], [0, 1, 2], [5, -1, -1]], np.int32)
    lens = np.array([20, 40, 0], np.int32)
    cap = pkv.load_library().pkv_shared_plan_max_ints(3, 8, 2, 48, 0)
    plan = pkv.plan_shared_prefix(bt, lens, 8, 2, 64, 16, 48)
    assert plan.host.size <= cap
    items, expected = check_coverage(plan, bt, lens, 4, 2)
    assert any(it[0] == 2 and not it[3] for it in items)
    assert expected[2] == 0
    # sequences 0 and 1 share block 0 and 1 but only 20 tokens -> below 32: no group
    assert all(it[1] == 4 for it in items)


def test_sharers_are_grouped_wherever_they_sit_in_the_batch():
    """Requests that reuse two cached prompts alternate in the batch with
    singletons: each prompt's requests form one group (its members listed in
    the items), and every token is still covered once."""
    bs, G = 16, 4
    rng = np.random.default_rng(3)
    prompt = {0: list(range(0, 20)), 1: list(range(20, 40))}      # 320 tokens each
    which = [0, 1, None, 0, 1, 0, None, 1, 0]
    next_block, rows, lens = 100, [], []
    for w_ in which:
        own_len = int(rng.integers(1, 60))
        base = prompt[w_] if w_ is not None else []
        L = len(base) * bs + own_len
        nb_own = -(-L // bs) - len(base)
        rows.append(base + list(range(next_block, next_block + nb_own)))
        next_block += nb_own
        lens.append(L)
    MB = max(len(r) for r in rows)
    bt = np.full((len(rows), MB), -1, np.int32)
    for i, r in enumerate(rows):
        bt[i, :len(r)] = r
    lens = np.array(lens, np.int32)
    plan = pkv.plan_shared_prefix(bt, lens, 16, 4, 128, bs, int(lens.max()), 256)
    items, expected = check_coverage(plan, bt, lens, G, 4)
    groups = {frozenset(it[7]) for it in items if it[1] > G}
    assert groups == {frozenset(i for i, w_ in enumerate(which) if w_ == p) for p in (0, 1)}
