// pkv_plan.cu -- host planner of the shared-prefix (cascade) decode path.
//
// Runs on the host, next to the block manager that owns the block tables:
// it finds runs of consecutive sequences whose tables start with the same
// physical block ids (forked samples, beams, a common system prompt), groups
// them, and cuts the attention work into items (cascade_plan.h).  The kernel
// side re-checks on the device that the members of a group really share the
// blocks it was told about.
#include <algorithm>
#include <cuda_runtime.h>
#include <cstring>
#include <vector>

#include "../../include/pkv.h"
#include "cascade_plan.h"

namespace {

// Smallest automatic item (tokens): below it the per-item fixed costs win.
constexpr int kMinAutoTokens = 64;

// SMs of the current device (the automatic cut targets three resident CTAs
// per SM); 152, a GB300's count, when no device answers.
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

struct Item {
    int seq0, nrows, slot;
    std::vector<Seg> segs;
    long long weight;  // tokens streamed, for the heavy-first order
    int entries;       // block-table entries of all segments
    std::vector<int> members;  // the sequences whose rows the item serves
};

int blocks_between(int tb, int te, int bs) { return (te + bs - 1) / bs - tb / bs; }

size_t split_total(long long seqs, long long heads, long long slots, long long head_dim)
{
    const size_t ml = (size_t)(seqs * heads * slots * 2) * sizeof(float);
    const size_t acc_off = (ml + 255) & ~size_t(255);
    return acc_off + (size_t)(seqs * heads * slots * head_dim) * sizeof(float);
}

}  // namespace

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
    // items per sequence: its partitions of at least P (or kMinAutoTokens)
    // tokens, one more for the rounding of a cut, one for a group's last item
    const int P = partition_size > 0 ? partition_size : kMinAutoTokens;
    const long long per_seq = (max_context_len + P - 1) / P + 2;
    return (size_t)pkv::plan::kHeader + 2 * (size_t)num_seqs +
           (size_t)(num_seqs * per_seq) * pkv::plan::item_ints(G);
}

int pkv_plan_shared_prefix(const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
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
    if (partition_size > 0 &&
        (partition_size % 32 || partition_size % block_size || partition_size / block_size > kTableCap / 4))
        return PKV_EINVAL;
    const int B = num_seqs, MB = max_blocks_per_seq, bs = block_size;
    const int align = bs > 32 ? bs : 32;
    const int max_members = kMaxRows / G;
    auto len_ok = [&](int s) {
        const int L = context_lens[s];
        return L > 0 && L <= max_context_len;
    };

    // Sequences that share leading blocks are grouped wherever they sit in
    // the batch (forked samples are neighbours, requests that reuse a cached
    // system prompt need not be): order them by the block ids of their
    // tables, valid contexts first and batch order among equal prefixes.
    auto nblk = [&](int s) { return len_ok(s) ? (context_lens[s] + bs - 1) / bs : 0; };
    std::vector<int> order(B);
    for (int s = 0; s < B; ++s)
        order[s] = s;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
        const int na = nblk(a), nb = nblk(b);
        if ((na > 0) != (nb > 0))
            return na > 0;
        const int32_t *ta = block_tables + (long long)a * MB, *tb = block_tables + (long long)b * MB;
        for (int j = 0, n = std::min(na, nb); j < n; ++j)
            if (ta[j] != tb[j])
                return ta[j] < tb[j];
        return false;
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
        int c = 0;
        while (c < n && a[c] == b[c])
            ++c;
        sp[k] = std::min(c * bs, std::min(la, lb)) / align * align;
    }

    // groups: runs of up to max_members neighbours in that order that share
    // S leading tokens (cnt == 1: a sequence on its own); member m of a
    // group is sequence order[first + m]
    struct Group {
        int first, cnt, S;
    };
    std::vector<Group> groups;
    long long total = 0;   // tokens to stream per kv head, shared ones once
    for (int k = 0; k < B;) {
        int cnt = 1, S = 0x7fffffff;
        while (cnt < max_members && k + cnt < B && sp[k + cnt] > 0) {
            S = std::min(S, sp[k + cnt]);
            ++cnt;
        }
        if (cnt < 2) {
            groups.push_back(Group{k, 1, 0});
            total += len_ok(order[k]) ? context_lens[order[k]] : 0;
        } else {
            groups.push_back(Group{k, cnt, S});
            total += S;
            for (int m = 0; m < cnt; ++m)
                total += context_lens[order[k + m]] - S;
        }
        k += cnt;
    }

    // A member's own tail costs whole 16-row loads; it joins its group's
    // last item while that item stays within T tokens (and within half the
    // block-id capacity), longer tails become items of their own.
    auto tail_cost = [](int t) { return (t + 15) / 16 * 16; };
    auto fold_tails = [&](const Group &g, int T, std::vector<char> *folded) {
        long long F = 0;
        int entries = 0;
        for (int m = 0; m < g.cnt; ++m) {
            const int t = context_lens[order[g.first + m]] - g.S, need = blocks_between(g.S, g.S + t, bs);
            const bool f = t > 0 && F + tail_cost(t) <= T && entries + need <= kTableCap / 2;
            if (f) {
                F += tail_cost(t);
                entries += need;
            }
            if (folded)
                (*folded)[m] = f;
        }
        return F;
    };
    // items per kv head that target T gives
    auto count_items = [&](int T) {
        long long n = 0;
        for (const Group &g : groups) {
            if (g.cnt == 1) {
                n += len_ok(order[g.first]) ? (context_lens[order[g.first]] + T - 1) / T : 1;
                continue;
            }
            std::vector<char> folded(g.cnt, 0);
            const long long F = fold_tails(g, T, &folded);
            n += std::max(1LL, (g.S + F + T - 1) / T);
            for (int m = 0; m < g.cnt; ++m) {
                const int t = context_lens[order[g.first + m]] - g.S;
                if (t > 0 && !folded[m])
                    n += (t + T - 1) / T;
            }
        }
        return n;
    };

    // Target tokens per item.  Automatic: the smallest T (a multiple of
    // `align`, between kMinAutoTokens or 4 blocks and 64 blocks) whose items
    // fit one CTA per resident slot of the GPU (three per SM) over all kv
    // heads, so that the launch runs as one wave of items of at most T tokens.
    int T = partition_size;
    if (T == 0) {
        const long long per_head = std::max(1LL, 3LL * gpu_sm_count() / num_kv_heads);
        const int lo = (std::max(4 * bs, kMinAutoTokens) + align - 1) / align;
        const int hi = (kTableCap / 4) * bs / align;
        int a = lo, b = hi;                       // in units of align
        while (a < b) {
            const int mid = (a + b) / 2;
            if (count_items(mid * align) <= per_head)
                b = mid;
            else
                a = mid + 1;
        }
        T = a * align;
    }

    std::vector<Item> items;
    std::vector<int> expected(B, 0);
    // [tb, te) cut into n nearly equal pieces at multiples of `align`
    auto cut = [&](int tb, int te, int n) {
        std::vector<int> b{tb};
        for (int i = 1; i < n; ++i) {
            const int x = (int)((tb + (long long)(te - tb) * i / n) / align * align);
            if (x > b.back() && x < te)
                b.push_back(x);
        }
        b.push_back(te);
        return b;
    };
    auto add_partitions = [&](int seq, int tb, int te, int first_slot) {
        const std::vector<int> b = cut(tb, te, (te - tb + T - 1) / T);
        for (size_t k = 0; k + 1 < b.size(); ++k)
            items.push_back(Item{seq, G, first_slot + (int)k, {Seg{seq, b[k], b[k + 1], 0, G}},
                                 (long long)(b[k + 1] - b[k]), blocks_between(b[k], b[k + 1], bs),
                                 {seq}});
        return (int)b.size() - 1;
    };

    for (const Group &g : groups) {
        const int s = order[g.first], cnt = g.cnt, S = g.S;
        std::vector<int> mem(order.begin() + g.first, order.begin() + g.first + cnt);
        if (cnt == 1) {
            if (!len_ok(s))
                items.push_back(Item{s, G, 0, {}, 0, 0, {s}});   // zero output
            else
                expected[s] = add_partitions(s, 0, context_lens[s], 0);
            continue;
        }
        // n_g items of at most about T tokens: the prefix cut into n_g - 1
        // equal pieces plus the part that goes with the folded tails
        const int rows = cnt * G;
        std::vector<char> folded(cnt, 0);
        const long long F = fold_tails(g, T, &folded);
        int n_g = (int)std::max(1LL, (S + F + T - 1) / T);
        int Sp = 0;
        if (n_g > 1) {
            const long long per = (S + F + n_g - 1) / n_g;
            const long long Pl = std::min<long long>(S, std::max(0LL, per - F));
            Sp = (int)((S - Pl) / align * align);
            if (Sp <= 0)
                n_g = 1, Sp = 0;
        }
        int n_pre = 0;
        if (n_g > 1) {
            const std::vector<int> b = cut(0, Sp, n_g - 1);
            for (size_t k = 0; k + 1 < b.size(); ++k, ++n_pre)
                items.push_back(Item{s, rows, n_pre, {Seg{s, b[k], b[k + 1], 0, rows}},
                                     (long long)(b[k + 1] - b[k]), blocks_between(b[k], b[k + 1], bs),
                                     mem});
        }
        Item last{s, rows, n_pre, {}, 0, 0, mem};
        if (Sp < S) {
            last.segs.push_back(Seg{s, Sp, S, 0, rows});
            last.weight += S - Sp;
            last.entries += blocks_between(Sp, S, bs);
        }
        for (int m = 0; m < cnt; ++m)
            if (folded[m]) {
                const int seq = mem[m], L = context_lens[seq];
                last.segs.push_back(Seg{seq, S, L, m * G, (m + 1) * G});
                last.weight += L - S;
                last.entries += blocks_between(S, L, bs);
            }
        items.push_back(last);
        const int n_items = n_pre + 1;
        for (int m = 0; m < cnt; ++m) {
            const int seq = mem[m], L = context_lens[seq];
            const int n_tail = (L > S && !folded[m]) ? add_partitions(seq, S, L, n_items) : 0;
            expected[seq] = n_items + n_tail;
        }
    }

    std::stable_sort(items.begin(), items.end(),
                     [](const Item &a, const Item &b) { return a.weight > b.weight; });
    int slots = 1;
    for (int s = 0; s < B; ++s)
        slots = std::max(slots, expected[s]);
    const int iints = item_ints(G);
    const size_t need = (size_t)kHeader + 2 * (size_t)B + items.size() * iints;
    if (plan_ints)
        *plan_ints = need;
    if (workspace_bytes)
        *workspace_bytes = split_total(B, num_heads, slots, head_dim);
    if (items.size() > 65535)
        return PKV_EUNSUPPORTED;
    if (!plan || plan_capacity_ints < need)
        return PKV_EWORKSPACE;

    for (const Item &it : items)
        if (it.entries > kTableCap)   // cannot happen: items are cut to fit
            return PKV_EUNSUPPORTED;
    std::memset(plan, 0, need * sizeof(int32_t));
    plan[H_NUM_ITEMS] = (int)items.size();
    plan[H_SLOTS] = slots;
    plan[H_NUM_SEQS] = B;
    plan[H_NUM_KV_HEADS] = num_kv_heads;
    plan[H_ITEM_INTS] = iints;
    plan[H_MAX_SEG] = max_segments(G);
    plan[H_PARTITION] = T;
    plan[H_TAG] = kTag;
    std::copy(expected.begin(), expected.end(), plan + kHeader);
    std::copy(context_lens, context_lens + B, plan + kHeader + B);
    int32_t *dst = plan + kHeader + 2 * (size_t)B;
    for (const Item &it : items) {
        const int nmem = it.nrows / G;
        int tiles = 0, nids = 0, checks = 0;
        dst[I_SEQ0] = it.seq0;
        for (int m = 0; m < kMaxRows; ++m)
            dst[kItemHead + m] = m < (int)it.members.size() ? it.members[m] : -1;
        dst[I_NROWS] = it.nrows;
        dst[I_SLOT] = it.slot;
        dst[I_NSEG] = (int)it.segs.size();
        int32_t *ids = dst + item_ids_offset(G);
        for (size_t k = 0; k < it.segs.size(); ++k) {
            const Seg &g = it.segs[k];
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
            for (int j = g.tok_begin / bs; j < (g.tok_end + bs - 1) / bs; ++j)
                *ids++ = row[j];
        }
        dst[I_TILES] = tiles;
        dst[I_IDS] = nids;
        dst[I_CHECKS] = checks;
        dst += iints;
    }
    return PKV_OK;
}

}  // extern "C"
