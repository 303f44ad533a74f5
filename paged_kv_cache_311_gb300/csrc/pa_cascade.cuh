// pa_cascade.cuh -- shared-prefix (cascade) decode attention.
//
// Sequences forked from one prompt (parallel sampling, beam search, a common
// system prompt) point their block tables at the same physical blocks for the
// shared part (PagedAttention: Efficient LLM Serving with vLLM, "Advanced
// Features", KV-Cache Sharing).  A per-sequence kernel reads those blocks once
// per sequence.  Here a host plan (cascade_plan.h) groups the sequences that
// share leading blocks and lays the work of one kv head out as a stream of
// 16-token tiles -- each group's shared prefix once for all members' query
// heads (up to 24 rows, three tensor-core n-tiles), then each member's own
// tail for that member's rows only, then the next group or ungrouped
// sequence -- cut into lists of nearly equal cost, one CTA per (kv head,
// list).  A list holds the pieces (items) of the groups its range covers;
// the CTA streams each item's segments through the same per-warp TMA rings
// and tensor-core engine as the per-sequence kernel, the rings' phases
// carrying over from item to item.  Rows of a sequence that one item holds
// entirely are written to the output directly; otherwise each item writes
// one partial per row and pa_cascade_merge_kernel, launched behind this
// kernel as a programmatic dependent (its CTAs take the SM slots this grid
// frees and wait for the grid to complete), merges them with log-sum-exp
// weights.
//
// Latency is what this kernel fights (each item streams only a few hundred
// tokens): the item carries its physical block ids, so the first TMA loads
// leave one round trip after the item is read, and the check of the device
// block tables and lengths and the q staging run while they fly.
#pragma once

#include "cascade_plan.h"
#include "pa_decode.cuh"
#include "pa_merge.cuh"

namespace pkv {

template <typename T, int D, int BS, int G>
struct CascadeCfg {
    using C = DecodeCfg<T, D, BS, G, true>;
    using Engine = TcEngine<T, D, BS, G, plan::kNT, true>;
    static constexpr int NW = C::NW, S = C::S;
    static constexpr int MAXSEG = plan::max_segments(G);
    static constexpr int ITEM_INTS = plan::item_ints(G);
    static constexpr int IDS = plan::item_ids_offset(G);
    static constexpr int SEGS = plan::item_segments_offset();
    static constexpr int TABLE_CAP = plan::kTableCap;
    // ring | barriers | flag | q rows | item copy (with its block ids) | bad
    // flag per segment, members' expected partial counts, a spare int and the
    // bad-length mask | per-row warp weights | the list's next item
    static constexpr int OFF_STAGES = 0;
    static constexpr int OFF_BAR = C::STAGES_BYTES;
    static constexpr int OFF_FLAG = OFF_BAR + NW * S * 8;
    static constexpr int OFF_Q = OFF_FLAG + 16;
    static constexpr int OFF_ITEM = OFF_Q + Engine::q_smem_bytes;
    static constexpr int EXTRA_INTS = ITEM_INTS + MAXSEG + plan::kMaxRows + 2;
    static constexpr int OFF_WTS = (OFF_ITEM + EXTRA_INTS * 4 + 15) / 16 * 16;
    static constexpr int OFF_NEXT = OFF_WTS + plan::kMaxRows * NW * 4;
    // the next-item buffer only where three CTAs per SM still fit (items of
    // many segments, small G, are larger)
    static constexpr bool PREFETCH = 3 * (OFF_NEXT + ITEM_INTS * 4 + 2048) <= 228 * 1024;
    static constexpr int SMEM_USED = OFF_NEXT + (PREFETCH ? ITEM_INTS * 4 : 0);
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;   // slack for 1024-byte alignment
    // three CTAs (12 warps) per SM: 228 KB of shared memory, 1 KB per CTA reserved
    static_assert(3 * (SMEM_BYTES + 1024) <= 228 * 1024, "three CTAs per SM");
    static_assert(OFF_Q % 16 == 0 && Engine::QROWB % 16 == 0, "q rows: 16-byte pieces");
    static_assert(C::TILE == plan::kTileTokens, "the planner counts the kernel's tiles");
};

template <typename T, int D, int BS, int G>
__global__ void __launch_bounds__(128, 3)
pa_cascade_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv, const int32_t *plan_buf)
{
    using CC = CascadeCfg<T, D, BS, G>;
    using C = typename CC::C;
    constexpr int NW = C::NW, S = C::S, TILE = C::TILE, NT = plan::kNT, RS = 8 * NT;
    constexpr int AWS = CC::Engine::AWS;
    static_assert(NW * RS * (AWS + 2) * 4 <= C::STAGES_BYTES, "merge scratch fits in the ring");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = aligned_smem(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kvh = blockIdx.x;
    init_rings<CC>(smem);

    // plan geometry from the launch: B fixes where the items start, the
    // slot count is the workspace's row stride
    const int B = p.num_seqs, slots = p.num_partitions;
    const int32_t *expected = plan_buf + plan::kHeader;
    const int32_t *plan_lens = expected + B;
    const int32_t *items = plan_buf + plan::kHeader + 2 * B;

    int32_t *it = reinterpret_cast<int32_t *>(smem + CC::OFF_ITEM);
    int32_t *segbad = it + CC::ITEM_INTS;    // segment k addresses a bad block
    int32_t *exp_s = segbad + CC::MAXSEG;    // expected partials per member
    // members whose device length differs from the plan's
    uint32_t *lenbad = reinterpret_cast<uint32_t *>(exp_s + plan::kMaxRows) + 1;
    uint32_t *cta_flag = reinterpret_cast<uint32_t *>(smem + CC::OFF_FLAG);
    if (tid == 0) {
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
        *cta_flag = 0;
    }
    float *mw = reinterpret_cast<float *>(smem + C::OFF_STAGES);
    float *lw = mw + NW * RS;
    float *aw = lw + NW * RS;
    float *wts = reinterpret_cast<float *>(smem + CC::OFF_WTS);   // [RS][NW]
    uint8_t *stages = smem + CC::OFF_STAGES + warp * S * C::STAGE_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + CC::OFF_BAR) + warp * S;
    // launched as a programmatic dependent of the previous kernel on the
    // stream: nothing that kernel may write is read before this wait.  Only
    // then may the merge kernel queued behind this grid start taking the
    // slots this grid frees (it waits for the whole grid before it reads
    // partials; the plan, which no kernel of this call writes, it reads
    // before that wait).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // The list's items one after the other.  `ring` counts the tiles this
    // warp has pushed through its ring so far (the stage and phase of the
    // next tile follow from it); a link that does not point further down the
    // item array ends the list, so the walk always ends.
    // Each item's record is fetched into a side buffer with asynchronous
    // copies while the item before it runs, and moved into place when that
    // item is done (the list's first item is read directly).
    int32_t *next_buf = reinterpret_cast<int32_t *>(smem + CC::OFF_NEXT);
    int ring = 0;
    bool fetched = false;
    for (int item = blockIdx.y; item >= 0 && item < p.num_items;) {
        if (tid == 0)
            *lenbad = 0;
        if (tid < CC::MAXSEG)
            segbad[tid] = 0;
        if (fetched) {
            cp_async_wait_all();
            __syncthreads();
            for (int i = tid; i < CC::ITEM_INTS; i += NW * 32)
                it[i] = next_buf[i];
        } else {
            // all loads in flight before the first store (see QRows)
            const int32_t *src = items + (int64_t)item * CC::ITEM_INTS;
            constexpr int PER = (CC::ITEM_INTS + NW * 32 - 1) / (NW * 32);
            int32_t v[PER];
#pragma unroll
            for (int u = 0; u < PER; ++u) {
                const int i = tid + u * NW * 32;
                v[u] = i < CC::ITEM_INTS ? src[i] : 0;
            }
#pragma unroll
            for (int u = 0; u < PER; ++u) {
                const int i = tid + u * NW * 32;
                if (i < CC::ITEM_INTS)
                    it[i] = v[u];
            }
        }
        __syncthreads();

        const int seq0 = it[plan::I_SEQ0], nrows = it[plan::I_NROWS], slot = it[plan::I_SLOT];
        const int nseg = it[plan::I_NSEG], total = it[plan::I_TILES];
        const int next = it[plan::I_NEXT] > item && it[plan::I_NEXT] < p.num_items ? it[plan::I_NEXT] : -1;
        fetched = CC::PREFETCH && next >= 0;
        if (fetched) {
            const int32_t *src = items + (int64_t)next * CC::ITEM_INTS;
            for (int i = tid; i < CC::ITEM_INTS; i += NW * 32)
                cp_async4(next_buf + i, src + i);
        }
        const int nmem = nrows / G;
        const int32_t *members = it + plan::kItemHead;   // the item's sequences, member m = rows mG..
        const CtaWork w{seq0, nrows, kvh, 0, 0, slot, seq0, members};
        if (nseg == 0) {  // empty or invalid context: zero rows, nothing to merge
            const int L = p.context_lens[seq0];
            if ((L < 0 || L > p.max_context_len) && tid == 0 && kvh == 0)
                report(p.status, PKV_DEV_BAD_CONTEXT_LEN);
            for (int idx = tid; idx < nrows * D; idx += blockDim.x)
                store_out(p.out, p.out_dtype, row_head(p, w, G, idx / D) * D + idx % D, 0.f);
            __syncthreads();
            item = next;
            continue;
        }
        // segment k: seg(k)[plan::S_*]; its block ids start at ids + S_ID_OFF
        auto seg = [&](int k) { return it + CC::SEGS + plan::kSegInts * k; };
        int32_t *ids = it + CC::IDS;
        // a list that timed out earlier streams nothing more: its remaining
        // items write failed rows
        const bool dead = *reinterpret_cast<volatile uint32_t *>(cta_flag) != 0;
        const bool invalid_item = it[plan::I_IDS] > CC::TABLE_CAP || nseg > CC::MAXSEG;

        // Segment of a tile.  Each warp asks for its tiles in increasing order,
        // separately for issuing and for consuming, so each keeps a cursor that
        // only moves forward.
        auto seg_of = [&](int tile, int &k) {
            while (k + 1 < nseg && seg(k + 1)[plan::S_FIRST_TILE] <= tile)
                ++k;
            return k;
        };
        const int my_n = invalid_item || dead ? 0 : (warp < total ? (total - 1 - warp) / NW + 1 : 0);
        int k_issue = 0, k_use = 0;
        // Issues tile i of this warp into stage st.  A block id outside the pool
        // invalidates its segment's rows (block 0 is loaded in its place).
        auto issue = [&](int i, int st) {
            const int tile = warp + i * NW, k = seg_of(tile, k_issue);
            const int *g = seg(k);
            const int tb = g[plan::S_BEGIN], te = g[plan::S_END], j0 = tb / BS;
            const int t0 = tb + (tile - g[plan::S_FIRST_TILE]) * TILE;
            uint8_t *kd = stages + st * C::STAGE_BYTES;
            uint8_t *vd = kd + C::TILE_BYTES;
            const int nbox = min(C::BOXES, (te - t0 + C::BOX_ROWS - 1) / C::BOX_ROWS);
            mbar_arrive_expect_tx(&bars[st], (uint32_t)(nbox * 2 * C::BOX_BYTES));
            for (int b = 0; b < nbox; ++b) {
                const int tok = t0 + b * C::BOX_ROWS;
                int phys = ids[g[plan::S_ID_OFF] + tok / BS - j0];
                if (phys < 0 || (int64_t)phys >= p.num_blocks) {
                    segbad[k] = 1;
                    phys = 0;
                }
                tma_load_5d(kd + b * C::BOX_BYTES, &tmk, &bars[st], 0, tok % BS, 0, kvh, phys);
                tma_load_5d(vd + b * C::BOX_BYTES, &tmv, &bars[st], 0, tok % BS, 0, kvh, phys);
            }
        };
        // ---- the item's small loads, then its first tiles: the device tables
        // must hold the plan's block ids (every member's table for a shared
        // prefix segment, the segment's own table otherwise); q rows to shared
        // memory; the members' expected partial counts and lengths.  The q
        // rows, the first 4 * NW * 32 table entries and the members' counts and
        // lengths are all requested before any of them is used, and before the
        // ring's tile loads, so that they do not queue behind a whole grid's
        // tiles: the start costs one round trip, and the tiles land while the
        // rows are stored.  An item with more entries to check takes more
        // rounds after it.
        const int vtotal = invalid_item ? 0 : it[plan::I_CHECKS];
        int got[4], want[4], kk[4];
        auto load_checks = [&](int x0) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int x = x0 + u * NW * 32 + tid;
                kk[u] = -1;
                got[u] = want[u] = 0;
                if (x < vtotal) {
                    int k = 0;
                    while (k + 1 < nseg && seg(k + 1)[plan::S_CHECK_OFF] <= x)
                        ++k;
                    const int *g = seg(k);
                    const int nb = (k + 1 < nseg ? seg(k + 1)[plan::S_ID_OFF] : it[plan::I_IDS]) -
                                   g[plan::S_ID_OFF];
                    const int local = x - g[plan::S_CHECK_OFF];
                    const int m = local / nb, i = local % nb;
                    const bool shared = g[plan::S_ROW_LO] == 0 && g[plan::S_ROW_HI] == nrows && nmem > 1;
                    const int s = shared ? members[m] : g[plan::S_TABLE_SEQ];
                    got[u] = p.block_tables[(int64_t)s * p.max_blocks_per_seq + g[plan::S_BEGIN] / BS + i];
                    want[u] = ids[g[plan::S_ID_OFF] + i];
                    kk[u] = k;
                }
            }
        };
        auto fold_checks = [&]() {
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (kk[u] >= 0 && got[u] != want[u])
                    segbad[kk[u]] = 1;
        };
        typename CC::Engine::QRows qrows;
        qrows.load(p, w);
        load_checks(0);
        int m_exp = 0, m_plen = 0, m_len = 0;
        if (tid < nmem) {
            const int sq = members[tid];
            m_exp = expected[sq];
            m_plen = plan_lens[sq];
            m_len = p.context_lens[sq];
        }
        if (lane == 0)
            for (int i = 0; i < (my_n < S ? my_n : S); ++i)
                issue(i, (ring + i) % S);
        fold_checks();
        qrows.store(smem + CC::OFF_Q);
        if (tid < nmem) {
            exp_s[tid] = m_exp;
            if (m_plen != m_len)
                atomicOr(lenbad, 1u << tid);
        }
        for (int x0 = 4 * NW * 32; x0 < vtotal; x0 += 4 * NW * 32) {
            load_checks(x0);
            fold_checks();
        }
        __syncthreads();

        if (!invalid_item && !dead) {
            typename CC::Engine eng;
            eng.init(p, smem + CC::OFF_Q, w, warp, lane);
            int failed_at = -1;
            for (int i = 0; i < my_n; ++i) {
                const int a = ring + i, st = a % S;
                if (!mbar_wait_bounded(&bars[st], (uint32_t)((a / S) & 1))) {
                    failed_at = i;
                    break;
                }
                const int tile = warp + i * NW, k = seg_of(tile, k_use);
                const int *g = seg(k);
                const int t0 = g[plan::S_BEGIN] + (tile - g[plan::S_FIRST_TILE]) * TILE;
                const int nvalid = min(TILE, g[plan::S_END] - t0);
                const uint32_t kbase = smem_u32(stages + st * C::STAGE_BYTES);
                eng.tile(kbase, kbase + C::TILE_BYTES, nvalid, lane, g[plan::S_ROW_LO], g[plan::S_ROW_HI]);
                __syncwarp();
                if (lane == 0 && i + S < my_n) {
                    fence_proxy_async_smem();
                    issue(i + S, st);
                }
            }
            if (failed_at >= 0) {
                const int last = min(my_n, failed_at + S);
                for (int i = failed_at; i < last; ++i) {
                    const int a = ring + i;
                    drain_wait(&bars[a % S], (uint32_t)((a / S) & 1), p.status);
                }
                if (lane == 0) {
                    report(p.status, PKV_DEV_TIMEOUT);
                    atomicOr(cta_flag, 1u);
                }
            }
            __syncthreads();
            eng.finish(mw, lw, aw, warp, lane, nrows);
        }
        ring += my_n;
        // The warps' (max, sum, acc) are in the scratch and every mark of a bad
        // block is in.
        __syncthreads();

        // ---- every row's result: the output itself for a sequence this item
        // holds entirely, otherwise this item's partial (read by the merge
        // through L2).  One thread per row finds whether the row fails -- a
        // segment serving it addresses a bad or disagreeing block id (marked by
        // the table check or by any issue of the loop), or its member's length
        // disagrees -- and folds the warps' (max, sum) into weights in shared
        // memory (1 / sum included for a final row); then float4 pieces of the
        // accumulators.
        const bool failed_all =
            invalid_item || *reinterpret_cast<volatile uint32_t *>(cta_flag) != 0;
        if (tid < nrows) {
            const int r = tid;
            const uint32_t lb = *lenbad;
            bool bad = failed_all || ((lb >> (r / G)) & 1u);
            for (int k = 0; k < nseg && k < CC::MAXSEG; ++k)
                bad = bad || (segbad[k] && r >= seg(k)[plan::S_ROW_LO] && r < seg(k)[plan::S_ROW_HI]);
            if (r == 0) {
                bool any = invalid_item;
                for (int k = 0; k < nseg && k < CC::MAXSEG; ++k)
                    any = any || segbad[k] != 0;
                if (any)
                    report(p.status, PKV_DEV_BAD_BLOCK);
                if (lb)
                    report(p.status, PKV_DEV_BAD_CONTEXT_LEN);
            }
            const bool final_row = exp_s[r / G] == 1;
            float M = -INFINITY, den = 0.f, f[NW];
#pragma unroll
            for (int k = 0; k < NW; ++k)
                M = fmaxf(M, bad ? -INFINITY : mw[k * RS + r]);
#pragma unroll
            for (int k = 0; k < NW; ++k) {
                const float mk = bad ? -INFINITY : mw[k * RS + r];
                f[k] = mk == -INFINITY ? 0.f : exp2f(mk - M);
                den += bad ? 0.f : f[k] * lw[k * RS + r];
            }
            const float norm = !final_row ? 1.f : (den > 0.f ? 1.f / den : 0.f);
#pragma unroll
            for (int k = 0; k < NW; ++k)
                wts[r * NW + k] = f[k] * norm;
            if (!final_row) {
                const int64_t base = row_head(p, w, G, r) * slots + slot;
                __stcg(reinterpret_cast<float2 *>(p.ws_ml) + base,
                       make_float2(bad ? -INFINITY : M, bad ? -1.f : den));
            }
        }
        __syncthreads();
        for (int idx = tid; idx < nrows * (D / 4); idx += blockDim.x) {
            const int r = idx / (D / 4), d4 = idx % (D / 4);
            float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < NW; ++k) {
                const float f = wts[r * NW + k];
                if (f != 0.f) {
                    const float4 a = reinterpret_cast<const float4 *>(aw + (k * RS + r) * AWS)[d4];
                    num.x += f * a.x;
                    num.y += f * a.y;
                    num.z += f * a.z;
                    num.w += f * a.w;
                }
            }
            const int64_t sh = row_head(p, w, G, r);
            if (exp_s[r / G] == 1) {
                store_out4(p.out, p.out_dtype, sh * D + 4 * d4, num);
            } else {
                __stcg(reinterpret_cast<float4 *>(p.ws_acc + (sh * slots + slot) * D) + d4, num);
            }
        }
        // the next item's loads overwrite the ring this item's epilogue used
        // as scratch: generic accesses first, then the async proxy's
        fence_proxy_async_smem();
        __syncthreads();
        item = next;
    }
}

// Merge of the shared-prefix partials, queued behind pa_cascade_kernel as a
// programmatic dependent: one half-warp per (sequence, head), eight per CTA.
// A plan gives a sequence only a few partials, so chunks of four slots keep
// the registers low enough for the whole grid to be resident at once.
// Sequences that one item held entirely (expected <= 1; 0 for an empty
// context) were written by pa_cascade_kernel itself.
template <int D>
__global__ void __launch_bounds__(128)
pa_cascade_merge_kernel(const __grid_constant__ DecodeParams p, const int32_t *plan_buf)
{
    const int hw = threadIdx.x >> 4, hl = threadIdx.x & 15;
    const int64_t sh = (int64_t)blockIdx.x * 8 + hw;
    const bool live = sh < (int64_t)p.num_seqs * p.num_heads;
    // the partial count comes from the plan, which the producing grid does
    // not write and which was complete before that grid passed its own wait
    const int n = live ? plan_buf[plan::kHeader + (int)(sh / p.num_heads)] : 0;
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the whole producing grid is done
    if (!live)
        return;
    merge_partials<D, 4>(p, sh, p.num_partitions, hl, [&]() { return n > 1 ? n : kMergeSkip; });
}

}  // namespace pkv
