"""The seeded workload generator: determinism and the block bookkeeping it
hands to the kernels, checked against the oracle's block manager rules."""
import numpy as np
import pytest

from oracle.block_manager import blocks_for_tokens
from workloads import CONFIGS, PagedDecodeWorkload, get


def _check_tables(w, inp):
    bs = w.bs
    tables, lens = inp.block_tables, inp.context_lens
    assert tables.shape == (w.num_seqs, w.max_blocks_per_seq)
    for s in range(w.num_seqs):
        n = blocks_for_tokens(int(lens[s]), bs)
        row = tables[s]
        assert (row[:n] >= 0).all() and (row[:n] < w.num_blocks).all()
        assert (row[n:] == -1).all()
        assert len(set(row[:n].tolist())) == n
    # slot of every new token is its sequence's block at pos // bs, offset pos % bs
    for sl, s, pos in zip(inp.slot_mapping, inp.token_seq, inp.token_pos):
        assert sl // bs == tables[s, pos // bs] and sl % bs == pos % bs
    # a physical block written this step belongs to exactly one sequence
    written = inp.slot_mapping // bs
    owners = {}
    for s in range(w.num_seqs):
        for b in tables[s][: blocks_for_tokens(int(lens[s]), bs)]:
            owners.setdefault(int(b), set()).add(s)
    for b in set(written.tolist()):
        assert len(owners[b]) == 1, "write into a block that is still shared"


@pytest.mark.parametrize("cfg", [c for c in CONFIGS if c.name != "long_context_bf16"],
                         ids=lambda c: c.name)
def test_generator_tables_follow_block_rules(cfg):
    w = PagedDecodeWorkload(cfg, 1234, total_steps=4)
    prev = w.context_lens().copy()
    for _ in range(4):
        inp = w.next_step()
        _check_tables(w, inp)
        if cfg.kind != "continuous":
            np.testing.assert_array_equal(inp.context_lens, prev + 1)
        prev = inp.context_lens.copy()
        assert inp.max_context_len == int(inp.context_lens.max())


def test_generator_is_deterministic():
    a = PagedDecodeWorkload(get(2), 7, total_steps=3)
    b = PagedDecodeWorkload(get(2), 7, total_steps=3)
    for _ in range(3):
        x, y = a.next_step(), b.next_step()
        np.testing.assert_array_equal(x.slot_mapping, y.slot_mapping)
        np.testing.assert_array_equal(x.block_tables, y.block_tables)


def test_shared_prefix_copy_on_write_pairs():
    cfg = get("shared_prefix_bf16")
    w = PagedDecodeWorkload(cfg, 31103, total_steps=2)
    partial = int(np.sum(w.prompt_lens % cfg.block_size != 0))
    first = w.next_step()
    assert first.cow_pairs.shape == (partial * (cfg.samples_per_prompt - 1), 2)
    assert len(set(first.cow_pairs[:, 1].tolist())) == first.cow_pairs.shape[0]
    assert not set(first.cow_pairs[:, 1].tolist()) & set(first.cow_pairs[:, 0].tolist())
    assert w.next_step().cow_pairs.shape[0] == 0
    # siblings still share every full prompt block
    t = first.block_tables
    for p, lp in enumerate(w.prompt_lens):
        full = int(lp) // cfg.block_size
        rows = t[p * 6:(p + 1) * 6, :full]
        assert (rows == rows[0]).all()


def test_continuous_batching_replaces_two_percent():
    cfg = get("llama13b_cb_bf16")
    w = PagedDecodeWorkload(cfg, 31102, total_steps=3)
    inp = w.next_step()
    B = w.num_seqs
    new_tokens = inp.num_tokens - B
    replaced = np.unique(inp.token_seq[:new_tokens])
    assert replaced.size == round(0.02 * B) == 5
    assert (inp.context_lens[replaced] >= 17).all() and (inp.context_lens[replaced] <= 513).all()


def test_long_context_pool_is_about_60_gb():
    cfg = get("long_context_bf16")
    for bs in (8, 16, 32):
        w = PagedDecodeWorkload(cfg.with_(block_size=bs), 31104, total_steps=1)
        pool_bytes = w.num_blocks * 2 * cfg.with_(block_size=bs).block_bytes
        assert 59e9 < pool_bytes <= 60e9
        assert w.init_lens.min() >= 16384 and w.init_lens.max() <= 32768


def test_system_prompt_requests_share_their_prompt_blocks_only():
    """Request i starts with system prompt i % 4 (1024-2048 tokens) and adds
    32-256 tokens of its own. The prompt's full blocks are held once, by
    exactly the requests on that prompt. Every other block is a single
    request's own."""
    cfg = get("system_prompt_bf16")
    w = PagedDecodeWorkload(cfg, 311 * 100 + 5, total_steps=3)
    inp = w.next_step()
    bs, B = cfg.block_size, w.num_seqs
    assert B == 256 and len(w.prompt_lens) == 4
    assert ((w.prompt_lens >= 1024) & (w.prompt_lens <= 2048)).all()
    np.testing.assert_array_equal(w.prompt_of, np.arange(B) % 4)
    own = inp.context_lens - w.prompt_lens[w.prompt_of]
    assert own.min() >= 32 + 1 and own.max() <= 256 + 1       # + the token of this step
    holders = {}
    for s in range(B):
        n = blocks_for_tokens(int(inp.context_lens[s]), bs)
        for j, b in enumerate(inp.block_tables[s, :n].tolist()):
            holders.setdefault(b, set()).add((s, j))
    for p in range(4):
        full = int(w.prompt_lens[p]) // bs
        members = [s for s in range(B) if s % 4 == p]
        first = inp.block_tables[members[0], :full]
        for s in members:
            np.testing.assert_array_equal(inp.block_tables[s, :full], first)
        for j, b in enumerate(first.tolist()):
            assert holders[b] == {(s, j) for s in members}
    shared = {int(b) for p in range(4)
              for b in inp.block_tables[p, :int(w.prompt_lens[p]) // bs].tolist()}
    for b, who in holders.items():
        if b not in shared:
            assert len(who) == 1, f"block {b} held by {who}"
    _check_tables(w, inp)


def test_llama_shaped_length_mixes():
    """Llama-7B-shaped batch: 64 sequences of U{128..2048} cached tokens.
    Llama-13B-shaped batch: 256 lengths round(600 e^(0.8 N)) clipped to
    [16, 4096], so the median sits near 600 and the tails reach the clips.
    Both add the token of the step."""
    w7 = PagedDecodeWorkload(get("llama7b_f16"), 311 * 100 + 1, total_steps=2)
    assert w7.num_seqs == 64
    assert w7.init_lens.min() >= 128 and w7.init_lens.max() <= 2048
    np.testing.assert_array_equal(w7.next_step().context_lens, w7.init_lens + 1)
    cfg13 = get("llama13b_cb_bf16")
    w13 = PagedDecodeWorkload(cfg13, 311 * 100 + 2, total_steps=2)
    L = w13.init_lens
    assert w13.num_seqs == 256 and L.min() >= 16 and L.max() <= 4096
    assert 450 <= np.median(L) <= 800
    # the log of the unclipped lengths has spread sigma = 0.8 around log 600
    inner = L[(L > 16) & (L < 4096)]
    assert 0.6 <= np.std(np.log(inner)) <= 1.0
