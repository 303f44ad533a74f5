// pkv_plan.cu -- host planner of the shared-prefix (cascade) decode path.
//
// Runs on the host, next to the block manager that owns the block tables:
// it brings together the sequences whose tables start with the same physical
// block ids (forked samples, beams, a common system prompt) wherever they sit
// in the batch, groups them, and cuts the attention work into items
// (cascade_plan.h).  The kernel side re-checks on the device that the members
// of a group really share the blocks it was told about.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/pkv.h"
#include "cascade_plan.h"

namespace {

// Smallest automatic list (tokens): below it the per-CTA fixed costs win.
constexpr int kMinAutoTokens = 64;
// Fewest tiles a list starts another unit with.
constexpr long long kMinPieceTiles = 4;

// SMs of the current device (the automatic cut targets one list per
// resident CTA of the shared-prefix kernel); 152, a GB300's count, when no
// device answers.
int gpu_sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();   // leave no error behind for the next launch check
        return 152;
    }
    return n;
}

struct Seg {
    int table_seq, tok_begin, tok_end, row_lo, row_hi;
};

// A work item; its segments and members live in flat arrays.
struct Item {
    int seq0, nrows, slot;
    int seg_begin, seg_count;   // in the segment array
    int mem_begin, mem_count;   // the sequences whose rows it serves: order[mem_begin ..]
    int entries;                // block-table entries of all segments
};

// First j < n with a[j] != b[j], else n.  Tables that share a long prefix
// (a cached prompt, forked samples) are compared 16 entries at a time.
int first_diff(const int32_t *a, const int32_t *b, int n)
{
    constexpr int kChunk = 16;
    int j = 0;
    if (n > 0 && a[0] != b[0])
        return 0;
    while (j + kChunk <= n && std::memcmp(a + j, b + j, kChunk * sizeof(int32_t)) == 0)
        j += kChunk;
    while (j < n && a[j] == b[j])
        ++j;
    return j;
}

int blocks_between(int tb, int te, int bs) { return (te + bs - 1) / bs - tb / bs; }

// Bytes of the split workspace (see DecodeParams): (max, sum) pairs, then the
// accumulators, 256-byte aligned.  False if the size does not fit in 64 bits.
bool split_total(uint64_t seqs, uint64_t heads, uint64_t slots, uint64_t head_dim, size_t *bytes)
{
    uint64_t rows, ml, acc;
    if (__builtin_mul_overflow(seqs, heads, &rows) || __builtin_mul_overflow(rows, slots, &rows) ||
        __builtin_mul_overflow(rows, (uint64_t)(2 * sizeof(float)), &ml) ||
        __builtin_mul_overflow(rows, head_dim * sizeof(float), &acc) || ml > UINT64_MAX - 256 ||
        ((ml + 255) & ~uint64_t(255)) > UINT64_MAX - acc)
        return false;
    *bytes = (size_t)(((ml + 255) & ~uint64_t(255)) + acc);
    return true;
}

// Longest context the planner takes: far beyond any cache, small enough
// that token and tile arithmetic stays inside int.
constexpr int kMaxContext = 1 << 30;

}  // namespace

namespace pkv {

namespace {
std::atomic<int> g_plan_engine{0};   // the engine choice (pkv_decode_set_engine)
constexpr int kTcgen05Engine = 3;
}  // namespace

void set_shared_plan_engine(int engine) { g_plan_engine.store(engine, std::memory_order_relaxed); }

// The tcgen05 kernel (head_dim 128) runs one CTA per SM and overlaps an
// item's epilogue with the next item's loads (a switch costs about one
// tile); the warp-level kernel runs three CTAs per SM and drains its rings
// at every switch (about 6 us, ten tiles, measured on a GB300).
int shared_ctas_per_sm(int head_dim)
{
    return head_dim == 128 && g_plan_engine.load(std::memory_order_relaxed) == kTcgen05Engine ? 1 : 3;
}

int shared_item_cost_tiles(int head_dim) { return shared_ctas_per_sm(head_dim) == 1 ? 1 : 10; }

}  // namespace pkv

extern "C" {

size_t pkv_shared_plan_max_ints(int num_seqs, int num_heads, int num_kv_heads, int max_context_len,
                                int partition_size)
{
    if (num_seqs <= 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads ||
        max_context_len < 0 || partition_size < 0)
        return 0;
    const int G = num_heads / num_kv_heads;
    if (G > pkv::plan::kMaxRows)
        return 0;
    // lists: at most the automatic count (one per resident CTA slot) or the
    // stream over the explicit target, or the stream over the smallest list
    // the table capacity allows (block size 8); items: every unit's first
    // piece (at most one per sequence) plus one more per list boundary
    using namespace pkv::plan;
    const long long W = (long long)num_seqs * (((long long)max_context_len + kTileTokens - 1) / kTileTokens);
    const long long q_cap = (long long)(kTableCap - 2 * max_segments(G)) * 8 / kTileTokens;
    long long lists = (W + q_cap - 1) / q_cap + 1;
    if (partition_size > 0)
        lists = std::max(lists, W / std::max(1, partition_size / kTileTokens) + 1);
    else
        lists = std::max(lists, 3LL * gpu_sm_count() / num_kv_heads + 1);   // the most CTAs per SM
    lists = std::min(lists, 65536LL);   // a plan never has more (PKV_EUNSUPPORTED)
    return (size_t)kHeader + 2 * (size_t)num_seqs +
           (size_t)(num_seqs + lists) * item_ints(G);
}

// The planner proper; pkv_plan_shared_prefix below only turns a failed host
// allocation into a status instead of an exception through the C ABI.
static int plan_shared_prefix(const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                              int max_blocks_per_seq, int block_size, int num_heads,
                              int num_kv_heads, int head_dim, int max_context_len,
                              int partition_size, int32_t *plan, size_t plan_capacity_ints,
                              size_t *plan_ints, size_t *workspace_bytes)
{
    using namespace pkv::plan;
    if (num_seqs <= 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads ||
        max_blocks_per_seq <= 0 || block_size <= 0 || max_context_len < 0 || partition_size < 0 ||
        head_dim <= 0 || !block_tables || !context_lens)
        return PKV_EINVAL;
    if ((long long)max_context_len > (long long)max_blocks_per_seq * block_size)
        return PKV_EINVAL;
    const int G = num_heads / num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return PKV_EUNSUPPORTED;
    // what the decode kernels take (the plan is made for them)
    if ((block_size != 8 && block_size != 16 && block_size != 32) || (head_dim != 64 && head_dim != 128) ||
        max_context_len > kMaxContext)
        return PKV_EUNSUPPORTED;
    if (partition_size > 0 &&
        (partition_size % 32 || partition_size % block_size || partition_size / block_size > kTableCap / 4))
        return PKV_EINVAL;
    const int B = num_seqs, MB = max_blocks_per_seq, bs = block_size;
    const int align = std::max(bs, kTileTokens);   // shared prefixes end on a tile and a block
    const int max_members = kMaxRows / G;
    auto len_ok = [&](int s) {
        const int L = context_lens[s];
        return L > 0 && L <= max_context_len;
    };

    // Sequences that share leading blocks are grouped wherever they sit in
    // the batch (forked samples are neighbours, requests that reuse a cached
    // system prompt need not be): order them by the block ids of their
    // tables, lexicographically (a table that is a prefix of another first),
    // valid contexts first and batch order among equal tables.
    auto nblk = [&](int s) { return len_ok(s) ? (context_lens[s] + bs - 1) / bs : 0; };
    std::vector<int> order(B);
    for (int s = 0; s < B; ++s)
        order[s] = s;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
        const int na = nblk(a), nb = nblk(b);
        if ((na > 0) != (nb > 0))
            return na > 0;
        const int32_t *ta = block_tables + (long long)a * MB, *tb = block_tables + (long long)b * MB;
        const int n = std::min(na, nb), j = first_diff(ta, tb, n);
        return j < n ? ta[j] < tb[j] : na < nb;
    });

    // tokens that order[k] shares with order[k - 1]
    std::vector<int> sp(B, 0);
    for (int k = 1; k < B; ++k) {
        const int sa = order[k - 1], sb = order[k];
        if (!len_ok(sa) || !len_ok(sb))
            continue;
        const int la = context_lens[sa], lb = context_lens[sb];
        const int n = std::min(nblk(sa), nblk(sb));
        const int32_t *a = block_tables + (long long)sa * MB;
        const int32_t *b = block_tables + (long long)sb * MB;
        const int c = first_diff(a, b, n);
        sp[k] = std::min(c * bs, std::min(la, lb)) / align * align;
    }

    // groups: runs of up to max_members neighbours in that order that share
    // S leading tokens (cnt == 1: a sequence on its own); member m of a
    // group is sequence order[first + m]
    struct Group {
        int first, cnt, S;
    };
    std::vector<Group> groups;
    for (int k = 0; k < B;) {
        int cnt = 1, S = 0x7fffffff;
        while (cnt < max_members && k + cnt < B && sp[k + cnt] > 0) {
            S = std::min(S, sp[k + cnt]);
            ++cnt;
        }
        groups.push_back(cnt < 2 ? Group{k, 1, 0} : Group{k, cnt, S});
        k += cnt;
    }
    std::vector<int> expected(B, 0);

    // ---- the tile stream of one kv head: unit after unit, a unit being a
    // group (its shared prefix once for all members' rows, then each
    // member's own tail for that member's rows) or an ungrouped sequence
    // (whole).  Costs count 16-token tiles, the kernel's unit of load.
    struct Part {
        int table_seq, tb, te, row_lo, row_hi;
        long long t0, tiles;   // place in the unit's stream
    };
    struct Unit {
        int seq0, nrows;
        int mem_begin, mem_count;   // members: order[mem_begin ..]
        int part_begin, part_end;   // in the part array
        long long t0, tiles;        // place in the kv head's stream
        int pieces;
    };
    auto tiles_of = [](int tb, int te) { return (long long)((te - tb + kTileTokens - 1) / kTileTokens); };
    std::vector<Unit> units;
    std::vector<Part> parts;
    std::vector<int> empty;   // order positions of sequences with an empty or invalid context
    units.reserve(groups.size());
    parts.reserve((size_t)B + groups.size());
    long long W = 0;
    for (const Group &g : groups) {
        const int s = order[g.first];
        if (g.cnt == 1 && !len_ok(s)) {
            empty.push_back(g.first);
            continue;
        }
        Unit u{s, g.cnt * G, g.first, g.cnt, (int)parts.size(), 0, W, 0, 0};
        auto add = [&](int seq, int tb, int te, int lo, int hi) {
            const long long t = tiles_of(tb, te);
            parts.push_back(Part{seq, tb, te, lo, hi, u.tiles, t});
            u.tiles += t;
        };
        if (g.cnt == 1) {
            add(s, 0, context_lens[s], 0, G);
        } else {
            add(s, 0, g.S, 0, u.nrows);
            for (int m = 0; m < g.cnt; ++m) {
                const int L = context_lens[order[g.first + m]];
                if (L > g.S)
                    add(order[g.first + m], g.S, L, m * G, (m + 1) * G);
            }
        }
        u.part_end = (int)parts.size();
        W += u.tiles;
        units.push_back(u);
    }

    // ---- lists: the stream cut into consecutive ranges, one CTA each (per
    // kv head), of nearly equal cost whatever the units' sizes.  A list's
    // cost is its tiles plus the item cost for every item after its first
    // (what the CTA's switch from one item to the next costs the kernel that
    // runs the plan); a list does not start another unit with less than
    // kMinPieceTiles of budget left (no sliver items).  Greedy filling under
    // a budget gives the fewest lists for that budget; the budget is the
    // smallest whose lists fit one per resident CTA of that kernel over the
    // kv heads (automatic), or the explicit target.  An item's block ids
    // stay within the kernel's table capacity whatever the segments'
    // alignment.
    const long long kItemCostTiles = pkv::shared_item_cost_tiles(head_dim);
    const long long q_cap = (long long)(kTableCap - 2 * max_segments(G)) * bs / kTileTokens;
    auto walk = [&](long long budget, std::vector<long long> *cuts) {
        long long pos = 0, n = 0;
        size_t u = 0;
        if (cuts)
            cuts->assign(1, 0);
        while (pos < W) {
            ++n;
            long long cost = 0;
            for (bool first = true; pos < W; first = false) {
                while (units[u].t0 + units[u].tiles <= pos)
                    ++u;
                const long long avail = units[u].t0 + units[u].tiles - pos;
                const long long extra = first ? 0 : kItemCostTiles;
                const long long room = budget - cost - extra;
                if (avail <= room) {
                    cost += extra + avail;
                    pos += avail;
                    continue;
                }
                if (!first && room < kMinPieceTiles)
                    break;
                pos += std::max(1LL, room);
                break;
            }
            if (cuts)
                cuts->push_back(pos);
        }
        return n;
    };
    long long Q;
    if (partition_size > 0) {
        Q = std::min<long long>(partition_size / kTileTokens, q_cap);
    } else {
        const long long N = std::max(1LL, (long long)pkv::shared_ctas_per_sm(head_dim) * gpu_sm_count() /
                                              num_kv_heads);
        long long lo = std::min(q_cap, std::max<long long>(kMinAutoTokens / kTileTokens, (W + N - 1) / N));
        long long hi = lo;
        while (hi < q_cap && walk(hi, nullptr) > N)
            hi = std::min(q_cap, 2 * hi);
        while (lo < hi) {
            const long long mid = (lo + hi) / 2;
            if (walk(mid, nullptr) <= N)
                hi = mid;
            else
                lo = mid + 1;
        }
        Q = hi;
    }
    std::vector<long long> cuts;
    const long long nl = walk(Q, &cuts);

    // items: the pieces of units that each list's range covers, in stream
    // order; a piece serves all its unit's rows, with the unit's parts (or
    // pieces of them) inside its range as segments
    std::vector<Item> store;
    std::vector<Seg> segs;
    std::vector<std::vector<int>> lists((size_t)std::max(1LL, nl));   // indices into store
    store.reserve(units.size() + (size_t)nl + empty.size());
    segs.reserve(parts.size() + 2 * (size_t)nl);
    {
        size_t u = 0;
        for (long long k = 0; k < nl; ++k) {
            while (u < units.size() && units[u].t0 + units[u].tiles <= cuts[k])
                ++u;
            for (size_t v = u; v < units.size() && units[v].t0 < cuts[k + 1]; ++v) {
                Unit &un = units[v];
                const long long a0 = std::max(cuts[k], un.t0) - un.t0;
                const long long b0 = std::min(cuts[k + 1], un.t0 + un.tiles) - un.t0;
                if (a0 >= b0)
                    continue;
                Item it{un.seq0, un.nrows, un.pieces++, (int)segs.size(), 0, un.mem_begin, un.mem_count, 0};
                for (int p = un.part_begin; p < un.part_end; ++p) {
                    const Part &pt = parts[(size_t)p];
                    const long long x = std::max(a0, pt.t0), y = std::min(b0, pt.t0 + pt.tiles);
                    if (x >= y)
                        continue;
                    const int tb = pt.tb + (int)((x - pt.t0) * kTileTokens);
                    const int te = std::min(pt.te, pt.tb + (int)((y - pt.t0) * kTileTokens));
                    segs.push_back(Seg{pt.table_seq, tb, te, pt.row_lo, pt.row_hi});
                    it.entries += blocks_between(tb, te, bs);
                }
                it.seg_count = (int)segs.size() - it.seg_begin;
                lists[(size_t)k].push_back((int)store.size());
                store.push_back(it);
            }
        }
    }
    for (size_t e = 0; e < empty.size(); ++e) {   // zero output, no loads: any list
        const int pos = empty[e];
        lists[e % lists.size()].push_back((int)store.size());
        store.push_back(Item{order[pos], G, 0, (int)segs.size(), 0, pos, 1, 0});
    }
    for (const Unit &un : units)
        for (int m = 0; m < un.mem_count; ++m)
            expected[order[un.mem_begin + m]] = un.pieces;

    // list k starts at item k; the rest follow, each list's items chained
    std::vector<int> items;   // plan position -> store index
    std::vector<int> next;
    items.reserve(store.size());
    for (auto &l : lists)
        items.push_back(l[0]);
    next.assign(items.size(), -1);
    next.reserve(store.size());
    for (size_t k = 0; k < lists.size(); ++k) {
        int prev = (int)k;
        for (size_t j = 1; j < lists[k].size(); ++j) {
            items.push_back(lists[k][j]);
            next.push_back(-1);
            next[(size_t)prev] = (int)items.size() - 1;
            prev = (int)items.size() - 1;
        }
    }
    const int T = (int)(Q * kTileTokens);
    int slots = 1;
    for (int s = 0; s < B; ++s)
        slots = std::max(slots, expected[s]);
    const int iints = item_ints(G);
    const size_t need = (size_t)kHeader + 2 * (size_t)B + items.size() * iints;
    if (plan_ints)
        *plan_ints = need;
    size_t ws_bytes = 0;
    if (!split_total((uint64_t)B, (uint64_t)num_heads, (uint64_t)slots, (uint64_t)head_dim, &ws_bytes))
        return PKV_EUNSUPPORTED;
    if (workspace_bytes)
        *workspace_bytes = ws_bytes;
    if (items.size() > INT32_MAX / 2 || lists.size() > 65535)
        return PKV_EUNSUPPORTED;
    if (!plan || plan_capacity_ints < need)
        return PKV_EWORKSPACE;

    for (const Item &it : store)
        if (it.entries > kTableCap)   // cannot happen: items are cut to fit
            return PKV_EUNSUPPORTED;
    std::memset(plan, 0, need * sizeof(int32_t));
    plan[H_NUM_LISTS] = (int)lists.size();
    plan[H_SLOTS] = slots;
    plan[H_NUM_SEQS] = B;
    plan[H_NUM_KV_HEADS] = num_kv_heads;
    plan[H_ITEM_INTS] = iints;
    plan[H_MAX_SEG] = max_segments(G);
    plan[H_TARGET] = T;
    plan[H_NUM_ITEMS] = (int)items.size();
    std::copy(expected.begin(), expected.end(), plan + kHeader);
    std::copy(context_lens, context_lens + B, plan + kHeader + B);
    int32_t *dst = plan + kHeader + 2 * (size_t)B;
    for (size_t i = 0; i < items.size(); ++i) {
        const Item &it = store[(size_t)items[i]];
        dst[I_NEXT] = next[i];
        const int nmem = it.nrows / G;
        int tiles = 0, nids = 0, checks = 0;
        dst[I_SEQ0] = it.seq0;
        for (int m = 0; m < kMaxRows; ++m)
            dst[kItemHead + m] = m < it.mem_count ? order[it.mem_begin + m] : -1;
        dst[I_NROWS] = it.nrows;
        dst[I_SLOT] = it.slot;
        dst[I_NSEG] = it.seg_count;
        int32_t *ids = dst + item_ids_offset(G);
        for (int k = 0; k < it.seg_count; ++k) {
            const Seg &g = segs[(size_t)(it.seg_begin + k)];
            const int nb = blocks_between(g.tok_begin, g.tok_end, bs);
            const bool shared = g.row_lo == 0 && g.row_hi == it.nrows && nmem > 1;
            int32_t *q = dst + item_segments_offset() + kSegInts * k;
            q[S_TABLE_SEQ] = g.table_seq;
            q[S_BEGIN] = g.tok_begin;
            q[S_END] = g.tok_end;
            q[S_ROW_LO] = g.row_lo;
            q[S_ROW_HI] = g.row_hi;
            q[S_FIRST_TILE] = tiles;
            q[S_ID_OFF] = nids;
            q[S_CHECK_OFF] = checks;
            tiles += (g.tok_end - g.tok_begin + kTileTokens - 1) / kTileTokens;
            nids += nb;
            checks += (shared ? nmem : 1) * nb;
            const int32_t *row = block_tables + (long long)g.table_seq * MB;
            ids = std::copy(row + g.tok_begin / bs, row + (g.tok_end + bs - 1) / bs, ids);
        }
        dst[I_TILES] = tiles;
        dst[I_IDS] = nids;
        dst[I_CHECKS] = checks;
        dst += iints;
    }
    return PKV_OK;
}

int pkv_plan_shared_prefix(const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                           int max_blocks_per_seq, int block_size, int num_heads,
                           int num_kv_heads, int head_dim, int max_context_len,
                           int partition_size, int32_t *plan, size_t plan_capacity_ints,
                           size_t *plan_ints, size_t *workspace_bytes)
{
    try {
        return plan_shared_prefix(block_tables, context_lens, num_seqs, max_blocks_per_seq,
                                  block_size, num_heads, num_kv_heads, head_dim, max_context_len,
                                  partition_size, plan, plan_capacity_ints, plan_ints,
                                  workspace_bytes);
    } catch (const std::bad_alloc &) {
        return PKV_EHOSTMEM;
    } catch (...) {   // a size no vector can hold (std::length_error)
        return PKV_EINVAL;
    }
}

}  // extern "C"
