// pkv_plan.cu -- host planner of the shared-prefix (cascade) decode path.
//
// Runs on the host, next to the block manager that owns the block tables:
// it finds runs of consecutive sequences whose tables start with the same
// physical block ids (forked samples, beams, a common system prompt), groups
// them, and cuts the attention work into items (cascade_plan.h).  The kernel
// side re-checks on the device that the members of a group really share the
// blocks it was told about.
#include <algorithm>
#include <cstring>
#include <vector>

#include "../../include/pkv.h"
#include "cascade_plan.h"

namespace {

constexpr int kDefaultPartition = 256;

struct Seg {
    int table_seq, tok_begin, tok_end, row_lo, row_hi;
};

struct Item {
    int seq0, nrows, slot;
    std::vector<Seg> segs;
    long long weight;  // tokens x row n-tiles, for the heavy-first order
    int entries;       // block-table entries of all segments
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
    const int P = partition_size > 0 ? partition_size : kDefaultPartition;
    const long long per_seq = (max_context_len + P - 1) / P + 1;
    return (size_t)pkv::plan::kHeader + (size_t)num_seqs + (size_t)num_seqs * num_kv_heads +
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
    const int P = partition_size > 0 ? partition_size : kDefaultPartition;
    if (P % 32 || P % block_size || P / block_size > kTableCap / 2)
        return PKV_EINVAL;
    const int B = num_seqs, MB = max_blocks_per_seq, bs = block_size;
    const int align = bs > 32 ? bs : 32;
    const int max_members = kMaxRows / G;
    auto len_ok = [&](int s) {
        const int L = context_lens[s];
        return L > 0 && L <= max_context_len;
    };

    // tokens sequence s shares with s - 1
    std::vector<int> sp(B, 0);
    for (int s = 1; s < B; ++s) {
        if (!len_ok(s - 1) || !len_ok(s))
            continue;
        const int la = context_lens[s - 1], lb = context_lens[s];
        const int n = std::min((la + bs - 1) / bs, (lb + bs - 1) / bs);
        const int32_t *a = block_tables + (long long)(s - 1) * MB;
        const int32_t *b = block_tables + (long long)s * MB;
        int c = 0;
        while (c < n && a[c] == b[c])
            ++c;
        sp[s] = std::min(c * bs, std::min(la, lb)) / align * align;
    }

    std::vector<Item> items;
    std::vector<int> expected(B, 0);
    auto add_partitions = [&](int seq, int tb, int te, int first_slot) {
        int k = 0;
        for (int t = tb; t < te; t += P, ++k) {
            const int e = std::min(t + P, te);
            items.push_back(Item{seq, G, first_slot + k, {Seg{seq, t, e, 0, G}}, (long long)(e - t),
                                 blocks_between(t, e, bs)});
        }
        return k;
    };

    for (int s = 0; s < B;) {
        int cnt = 1, S = 0x7fffffff;
        while (cnt < max_members && s + cnt < B && sp[s + cnt] > 0) {
            S = std::min(S, sp[s + cnt]);
            ++cnt;
        }
        if (cnt < 2) {                       // a sequence on its own
            if (!len_ok(s)) {
                items.push_back(Item{s, G, 0, {}, 0, 0});   // zero output
            } else {
                expected[s] = add_partitions(s, 0, context_lens[s], 0);
            }
            s += 1;
            continue;
        }
        // a group [s, s + cnt) sharing S tokens
        const int rows = cnt * G;
        const int first_item = (int)items.size();
        const int n_pre = (S + P - 1) / P;
        for (int x = 0; x < n_pre; ++x) {
            const int t = x * P, e = std::min(t + P, S);
            items.push_back(Item{s, rows, x, {Seg{s, t, e, 0, rows}}, (long long)(e - t) * 3,
                                 blocks_between(t, e, bs)});
        }
        for (int m = 0; m < cnt; ++m) {
            const int seq = s + m, L = context_lens[seq];
            int n_tail = 0;
            if (L > S) {
                Item &last = items[first_item + n_pre - 1];
                const int need = blocks_between(S, L, bs);
                if (L - S <= P && last.entries + need <= kTableCap) {
                    last.segs.push_back(Seg{seq, S, L, m * G, (m + 1) * G});
                    last.weight += L - S;
                    last.entries += need;
                } else {
                    n_tail = add_partitions(seq, S, L, n_pre);
                }
            }
            expected[seq] = n_pre + n_tail;
        }
        s += cnt;
    }

    std::stable_sort(items.begin(), items.end(),
                     [](const Item &a, const Item &b) { return a.weight > b.weight; });
    int slots = 1;
    for (int s = 0; s < B; ++s)
        slots = std::max(slots, expected[s]);
    const int iints = item_ints(G);
    const size_t need = (size_t)kHeader + B + (size_t)B * num_kv_heads + items.size() * iints;
    if (plan_ints)
        *plan_ints = need;
    if (workspace_bytes)
        *workspace_bytes = split_total(B, num_heads, slots, head_dim);
    if (items.size() > 65535)
        return PKV_EUNSUPPORTED;
    if (!plan || plan_capacity_ints < need)
        return PKV_EWORKSPACE;

    std::memset(plan, 0, need * sizeof(int32_t));
    plan[H_NUM_ITEMS] = (int)items.size();
    plan[H_SLOTS] = slots;
    plan[H_NUM_SEQS] = B;
    plan[H_NUM_KV_HEADS] = num_kv_heads;
    plan[H_ITEM_INTS] = iints;
    plan[H_MAX_SEG] = max_segments(G);
    plan[H_PARTITION] = P;
    plan[H_TAG] = kTag;
    std::copy(expected.begin(), expected.end(), plan + kHeader);
    int32_t *dst = plan + kHeader + B + (size_t)B * num_kv_heads;
    for (const Item &it : items) {
        dst[0] = it.seq0;
        dst[1] = it.nrows;
        dst[2] = it.slot;
        dst[3] = (int)it.segs.size();
        for (size_t k = 0; k < it.segs.size(); ++k) {
            const Seg &g = it.segs[k];
            int32_t *q = dst + kItemHead + kSegInts * k;
            q[0] = g.table_seq;
            q[1] = g.tok_begin;
            q[2] = g.tok_end;
            q[3] = g.row_lo;
            q[4] = g.row_hi;
        }
        dst += iints;
    }
    return PKV_OK;
}

}  // extern "C"
