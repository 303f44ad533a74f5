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


def plan_lists(plan, B):
    """The plan's work lists: list k starts at item k and follows the
    items' next links, which only point further down; every item belongs to
    exactly one list."""
    h = plan.host
    n_lists, iints, n_items = int(h[0]), int(h[4]), int(h[7])
    assert (plan.num_lists, plan.num_items) == (n_lists, n_items)
    assert 1 <= n_lists <= n_items
    base = 8 + 2 * B
    seen, lists = set(), []
    for k in range(n_lists):
        chain, i = [], k
        while i >= 0:
            assert i not in seen
            seen.add(i)
            chain.append(i)
            nxt = int(h[base + i * iints + 7])
            assert nxt == -1 or i < nxt < n_items
            i = nxt
        lists.append(chain)
    assert seen == set(range(n_items))
    return lists


def list_tiles(plan, B):
    h, iints = plan.host, int(plan.host[4])
    return [sum(int(h[8 + 2 * B + i * iints + 4]) for i in chain) for chain in plan_lists(plan, B)]


ITEM_COST = 10       # tiles a CTA's switch to its list's next item costs the planner
MIN_PIECE = 4        # fewest tiles a list starts another unit with


def list_costs(plan, B):
    """A list's cost as the planner balances it: its tiles plus ITEM_COST
    for every item after the first that streams tiles (the zero-output items
    of empty contexts are appended outside the balanced stream)."""
    h, iints = plan.host, int(plan.host[4])
    costs = []
    for t, chain in zip(list_tiles(plan, B), plan_lists(plan, B)):
        n = sum(1 for i in chain if int(h[8 + 2 * B + i * iints + 4]) > 0)
        costs.append(t + ITEM_COST * max(0, n - 1))
    return costs


def check_budget(plan, B):
    """Every list costs at most the plan's budget, and the greedy fill leaves
    no list but the last one far below it (a list ends only when the next
    unit would start with less than MIN_PIECE tiles after its item cost, or
    at the budget itself inside a unit)."""
    budget = int(plan.host[6]) // 16
    costs = list_costs(plan, B)
    assert max(costs) <= budget
    assert min(costs[:-1], default=budget) >= budget - ITEM_COST - MIN_PIECE
    return budget, costs


def decode_plan(plan, B, Hk, G):
    h = plan.host
    n_lists, slots, nseq, nkv, iints, maxseg, target, n_items = (int(x) for x in h[:8])
    assert (nseq, nkv) == (B, Hk)
    plan_lists(plan, B)
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
    # an item writes one partial per row of every member it lists (an empty
    # one for a member none of its segments serve), in its slot: each
    # (sequence, slot) exactly once, slots 0 .. expected - 1
    slots_seen = [[] for _ in range(B)]
    for seq0, nrows, slot, segs, ids, totals, raw, members in items:
        assert len(set(members)) == len(members)
        assert nrows % G == 0 and nrows <= 24 and len(members) == nrows // G
        if not segs:
            assert lens[seq0] <= 0
            continue
        for s in members:
            slots_seen[s].append(slot)
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
    for s in range(B):
        if lens[s] > 0:
            assert (covered[s] == 1).all(), f"sequence {s} not covered exactly once"
            assert sorted(slots_seen[s]) == list(range(int(expected[s])))
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
        shared = int(lp) // 16 * 16           # the prompt's full blocks
        mine = [it for it in prefix_items if set(it[7]) == set(range(6 * p, 6 * p + 6))]
        assert sum(seg[2] - seg[1] for it in mine for seg in it[3] if seg[3] == 0 and seg[4] == 24) == shared


def stream_tiles(items):
    """Tiles of the per-kv-head stream: every item's segments, 16 tokens a tile."""
    return sum(-(-(te - tb) // 16) for it in items for _, tb, te, _, _ in it[3])


@pytest.mark.parametrize("name,step", [("shared_prefix_bf16", 6), ("shared_prefix_bf16", 120),
                                       ("system_prompt_bf16", 30)])
def test_automatic_plan_is_one_balanced_wave(name, step):
    """partition_size 0: one list per resident CTA slot (3 per SM; 152 SMs
    when no GPU answers) over the kv heads, each list within a snap (at most
    8 tiles) of an equal share of the stream, whatever the groups' sizes."""
    cfg = get(name)
    w = PagedDecodeWorkload(cfg, 31103, total_steps=step + 2)
    for _ in range(step + 1):
        inp = w.next_step()
    plan = pkv.plan_shared_prefix(inp.block_tables, inp.context_lens, cfg.num_heads, cfg.num_kv_heads,
                                  cfg.head_dim, cfg.block_size, inp.max_context_len)
    items, expected = check_coverage(plan, inp.block_tables, inp.context_lens, cfg.group,
                                     cfg.num_kv_heads)
    B = len(inp.context_lens)
    tiles = list_tiles(plan, B)
    W = stream_tiles(items)
    assert sum(tiles) == W
    n, N = len(tiles), 3 * 152 // cfg.num_kv_heads
    assert N - 2 <= n <= N
    budget, costs = check_budget(plan, B)
    # the budget pays for the item switches the cuts need, not much more
    assert -(-W // N) <= budget <= -(-W // N) + ITEM_COST + MIN_PIECE
    # a piece per list boundary at most: items <= units + lists - 1
    assert len(items) <= len({frozenset(it[7]) for it in items}) + n - 1


def test_no_sharing_gives_equal_lists_of_whole_sequences():
    cfg = get("llama7b_f16")
    inp = PagedDecodeWorkload(cfg, 1, total_steps=1).next_step()
    plan = pkv.plan_shared_prefix(inp.block_tables, inp.context_lens, 32, 32, 128, 16,
                                  inp.max_context_len, 512)
    items, expected = check_coverage(plan, inp.block_tables, inp.context_lens, 1, 32)
    assert all(it[1] == 1 and len(it[3]) == 1 for it in items)
    # lists of a 512-token (32-tile) budget over the stream of all sequences
    tiles = list_tiles(plan, len(inp.context_lens))
    W = int((-(-inp.context_lens // 16)).sum())
    assert sum(tiles) == W
    budget, _ = check_budget(plan, len(inp.context_lens))
    assert budget == 32
    assert expected.sum() == len(items)


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
    # the first group streams 192 shared tokens, five 13-token tails (a tile
    # each) and one 708-token tail: 12 + 5 + 45 = 62 tiles over 16-tile
    # lists, so its members take at least four partials each
    assert all(expected[m] >= 4 for m in range(6))
    assert check_budget(plan, 8)[0] == 16


def test_empty_context_gets_a_zero_item_and_plan_size_is_bounded():
    bt = np.array([[0, 1, -1], [0, 1, 2], [5, -1, -1]], np.int32)
    lens = np.array([20, 40, 0], np.int32)
    cap = pkv.load_library().pkv_shared_plan_max_ints(3, 8, 2, 48, 0)
    plan = pkv.plan_shared_prefix(bt, lens, 8, 2, 64, 16, 48)
    assert plan.host.size <= cap
    items, expected = check_coverage(plan, bt, lens, 4, 2)
    assert any(it[0] == 2 and not it[3] for it in items)
    assert expected[2] == 0
    # sequences 0 and 1 share blocks 0 and 1, but sequence 0 holds only 20
    # tokens: their shared prefix is its first full 16-token tile
    pre = [seg for it in items for seg in it[3] if it[1] == 8 and seg[3] == 0 and seg[4] == 8]
    assert sum(te - tb for _, tb, te, _, _ in pre) == 16


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


def random_batch(rng, prefix_rate=0.0):
    """A few prompts forked into members with random tails, singletons and
    empty contexts, in shuffled batch order.  With prefix_rate, a member's
    context may end inside its prompt: its table is then a prefix of the
    prompt's shared blocks (plus its own copy of a partial block)."""
    bs = int(rng.choice([8, 16, 32]))
    rows, lens, nxt = [], [], 0
    for _ in range(int(rng.integers(1, 5))):           # forked prompts
        P_ = int(rng.integers(1, 700))
        full, rem = divmod(P_, bs)
        shared = list(range(nxt, nxt + full))
        nxt += full
        for _m in range(int(rng.integers(1, 9))):
            if rng.random() < prefix_rate:
                L = int(rng.integers(1, P_ + 1))
            else:
                L = P_ + int(rng.integers(0, 200))
            nb = -(-L // bs)
            own = max(0, nb - full)
            rows.append(shared[:nb] + list(range(nxt, nxt + own)))
            nxt += own
            lens.append(L)
    for _ in range(int(rng.integers(0, 4))):           # singletons and empty contexts
        L = int(rng.integers(0, 400))
        nb = -(-L // bs)
        rows.append(list(range(nxt, nxt + nb)))
        nxt += nb
        lens.append(L)
    order = rng.permutation(len(rows))
    rows = [rows[i] for i in order]
    lens = np.array([lens[i] for i in order], np.int32)
    MB = max(1, max(len(r) for r in rows))
    bt = np.full((len(rows), MB), -1, np.int32)
    for i, r in enumerate(rows):
        bt[i, :len(r)] = r
    return bs, bt, lens


def check_random_batch(rng, prefix_rate):
    bs, bt, lens = random_batch(rng, prefix_rate)
    G = int(rng.choice([1, 2, 4, 8]))
    Hk = int(rng.integers(1, 4))
    # automatic, or an explicit target: a multiple of 32 and of bs, at most 64 blocks
    target = int(rng.choice([0, 0, max(bs, 32) * int(rng.integers(1, 9))]))
    mcl = max(int(lens.max()), 1)
    plan = pkv.plan_shared_prefix(bt, lens, G * Hk, Hk, 128, bs, mcl, target)
    assert plan.host.size <= pkv.load_library().pkv_shared_plan_max_ints(len(lens), G * Hk, Hk, mcl, target)
    items, expected = check_coverage(plan, bt, lens, G, Hk, bs=bs)
    if items and any(it[3] for it in items):
        budget, costs = check_budget(plan, len(lens))
        if target:
            assert budget <= target // 16    # the explicit target caps every list's cost


@pytest.mark.parametrize("seed", range(24))
def test_random_batches_cover_exactly_within_budget(seed):
    """Random batches, block size, query group and target: every token is
    covered once per query row, lists are well formed and within their
    budget, and the plan fits the size bound."""
    check_random_batch(np.random.default_rng(1000 + seed), 0.0)


@pytest.mark.parametrize("seed", range(24))
def test_random_batches_with_prefix_tables(seed):
    """As above, with members whose context ends inside their prompt, so
    that some tables are prefixes of others (the ordering that brings
    sharers together is then still a strict one)."""
    check_random_batch(np.random.default_rng(2000 + seed), 0.3)


def test_prefix_table_sorts_before_its_extensions():
    """A table that is a prefix of others (a request whose context ends
    inside a cached prompt) is ordered before them and grouped with them,
    wherever it sits in the batch: the group's shared part is the prefix's
    full blocks."""
    bs = 16
    prompt = list(range(10))                       # 160 tokens of cached prompt
    rows = [prompt + [100], prompt[:4], prompt + [101], list(range(200, 203)), prompt + [102]]
    lens = np.array([161, 64, 170, 40, 175], np.int32)
    bt = np.full((len(rows), 11), -1, np.int32)
    for i, r in enumerate(rows):
        bt[i, :len(r)] = r
    plan = pkv.plan_shared_prefix(bt, lens, 8, 2, 128, bs, int(lens.max()), 0)
    items, _ = check_coverage(plan, bt, lens, 4, 2, bs=bs)
    grouped = [it for it in items if len(it[7]) > 1]
    assert grouped and {frozenset(it[7]) for it in grouped} == {frozenset({1, 0, 2, 4})}
    # the group lists the prefix's sequence first and shares its 64 tokens
    assert all(it[7][0] == 1 for it in grouped)
    shared = [seg for it in grouped for seg in it[3] if seg[3] == 0 and seg[4] == it[1]]
    assert shared and max(seg[2] for seg in shared) == 64


def test_too_many_lists_is_refused():
    """An explicit target far too small for the batch would need more lists
    than a grid's y extent (65,535): the planner refuses it."""
    bs, B, L = 16, 512, 4096                      # 256 tiles each, no sharing
    bt = np.arange(B * (L // bs), dtype=np.int32).reshape(B, L // bs)
    lens = np.full(B, L, np.int32)
    with pytest.raises(pkv.PkvError) as e:
        pkv.plan_shared_prefix(bt, lens, 4, 1, 128, bs, L, 32)   # 2 tiles per list: 65,536 lists
    assert e.value.status == -2
    plan = pkv.plan_shared_prefix(bt, lens, 4, 1, 128, bs, L, 64)   # 4 tiles per list: 32,768
    assert plan.num_lists == B * 256 // 4
