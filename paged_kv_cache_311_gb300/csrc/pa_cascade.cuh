// pa_cascade.cuh -- shared-prefix (cascade) decode attention.
//
// Sequences forked from one prompt (parallel sampling, beam search, a common
// system prompt) point their block tables at the same physical blocks for the
// shared part (PagedAttention: Efficient LLM Serving with vLLM, "Advanced
// Features", KV-Cache Sharing).  A per-sequence kernel reads those blocks once
// per sequence.  Here a host plan (cascade_plan.h) groups consecutive sequences
// that share leading blocks and cuts the work into items; one CTA per (kv
// head, item) streams the item's segments -- a partition of the shared prefix
// for every member's query heads (up to 24 rows, three tensor-core n-tiles),
// plus, in a group's last item, each member's own tail for that member's rows
// only -- through the same per-warp TMA rings and tensor-core engine as the
// per-sequence kernel.  Each item writes one partial per row; the CTA that
// delivers a sequence's last partial (counted with one atomic per (sequence,
// kv head)) merges that sequence's partials with log-sum-exp weights and
// writes its output, so no separate merge kernel runs.
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
    static constexpr int TABLE_CAP = plan::kTableCap;
    // ring | barriers | flag | q rows | block table | item copy, first tile /
    // table offset / bad flag per segment, merge flags | per-row warp weights
    static constexpr int OFF_STAGES = 0;
    static constexpr int OFF_BAR = C::STAGES_BYTES;
    static constexpr int OFF_FLAG = OFF_BAR + NW * S * 8;
    static constexpr int OFF_Q = OFF_FLAG + 16;
    static constexpr int OFF_TABLE = OFF_Q + Engine::q_smem_bytes;
    static constexpr int OFF_EXTRA = OFF_TABLE + TABLE_CAP * 4;
    static constexpr int EXTRA_INTS = ITEM_INTS + 3 * (MAXSEG + 1) + plan::kMaxRows;
    static constexpr int OFF_WTS = (OFF_EXTRA + EXTRA_INTS * 4 + 15) / 16 * 16;
    static constexpr int SMEM_USED = OFF_WTS + plan::kMaxRows * NW * 4;
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;   // slack for 1024-byte alignment
    // three CTAs (12 warps) per SM: 228 KB of shared memory, 1 KB per CTA reserved
    static_assert(3 * (SMEM_BYTES + 1024) <= 228 * 1024, "three CTAs per SM");
    static_assert(OFF_Q % 16 == 0 && Engine::QROWB % 16 == 0, "q rows: 16-byte pieces");
};

template <typename T, int D, int BS, int G>
__global__ void __launch_bounds__(128, 3)
pa_cascade_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv, int32_t *plan_buf)
{
    using CC = CascadeCfg<T, D, BS, G>;
    using C = typename CC::C;
    constexpr int NW = C::NW, S = C::S, TILE = C::TILE, NT = plan::kNT, RS = 8 * NT;
    static_assert(NW * RS * (D + 2) * 4 <= C::STAGES_BYTES, "merge scratch fits in the ring");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = aligned_smem(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kvh = blockIdx.x, item = blockIdx.y;

    const int B = plan_buf[plan::H_NUM_SEQS];
    const int Hk = plan_buf[plan::H_NUM_KV_HEADS];
    const int slots = plan_buf[plan::H_SLOTS];
    const int32_t *expected = plan_buf + plan::kHeader;
    int32_t *counters = plan_buf + plan::kHeader + B;
    const int32_t *src = plan_buf + plan::kHeader + B + (int64_t)B * Hk + (int64_t)item * CC::ITEM_INTS;

    int32_t *it = reinterpret_cast<int32_t *>(smem + CC::OFF_EXTRA);
    int32_t *first = it + CC::ITEM_INTS;     // first tile of segment k (k <= nseg)
    int32_t *tab = first + CC::MAXSEG + 1;   // table offset of segment k
    int32_t *segbad = tab + CC::MAXSEG + 1;  // segment k addresses a bad block
    int32_t *flag = segbad + CC::MAXSEG + 1; // merge flags per member
    for (int i = tid; i < CC::ITEM_INTS; i += blockDim.x)
        it[i] = src[i];
    init_rings<CC>(smem);
    __syncthreads();

    const int seq0 = it[0], nrows = it[1], slot = it[2], nseg = it[3];
    const int nmem = nrows / G;
    const CtaWork w{seq0, nrows, kvh, 0, 0, slot, seq0};
    if (nseg == 0) {  // empty or invalid context: zero rows, nothing to merge
        const int L = p.context_lens[seq0];
        if ((L < 0 || L > p.max_context_len) && tid == 0 && kvh == 0)
            report(p.status, PKV_DEV_BAD_CONTEXT_LEN);
        for (int idx = tid; idx < nrows * D; idx += blockDim.x)
            store_out(p.out, p.out_dtype, row_head(p, w, G, idx / D) * D + idx % D, 0.f);
        return;
    }
    const int *seg = it + plan::kItemHead;   // {table_seq, tok_begin, tok_end, row_lo, row_hi}
    if (tid == 0) {
        int tiles = 0, entries = 0;
        for (int k = 0; k < nseg; ++k) {
            first[k] = tiles;
            tab[k] = entries;
            segbad[k] = 0;
            const int b = seg[5 * k + 1], e = seg[5 * k + 2];
            tiles += (e - b + TILE - 1) / TILE;
            entries += (e + BS - 1) / BS - b / BS;
        }
        first[nseg] = tiles;
        tab[nseg] = entries;
    }
    __syncthreads();

    // ---- stage every segment's block-table slice; the members of a shared
    // prefix must hold the same block ids there (checked)
    int32_t *table_s = reinterpret_cast<int32_t *>(smem + CC::OFF_TABLE);
    uint32_t *cta_flag = reinterpret_cast<uint32_t *>(smem + CC::OFF_FLAG);
    // A bad block id (or a member whose shared blocks differ) invalidates the
    // rows of its segment only; block 0 is loaded in its place.
    const bool invalid_item = tab[nseg] > CC::TABLE_CAP;
    for (int k = 0; k < nseg && !invalid_item; ++k) {
        const int tseq = seg[5 * k], j0 = seg[5 * k + 1] / BS;
        const int nb = tab[k + 1] - tab[k];
        const int32_t *bt = p.block_tables + (int64_t)tseq * p.max_blocks_per_seq + j0;
        const bool shared_seg = seg[5 * k + 3] == 0 && seg[5 * k + 4] == nrows && nmem > 1;
        for (int i = tid; i < nb; i += blockDim.x) {
            int b = bt[i];
            bool bad = b < 0 || (int64_t)b >= p.num_blocks;
            if (shared_seg)
                for (int m = 1; m < nmem; ++m)
                    bad |= bt[(int64_t)m * p.max_blocks_per_seq + i] != b;
            if (bad) {
                segbad[k] = 1;
                b = 0;
            }
            table_s[tab[k] + i] = (b < 0 || (int64_t)b >= p.num_blocks) ? 0 : b;
        }
    }
    CC::Engine::stage_q_rows(p, smem + CC::OFF_Q, w);
    if (tid == 0) {
        *cta_flag = 0;
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
    }
    __syncthreads();
    if (tid == 0) {
        bool any = invalid_item;
        for (int k = 0; k < nseg; ++k)
            any |= segbad[k] != 0;
        if (any)
            report(p.status, PKV_DEV_BAD_BLOCK);
    }
    auto row_bad = [&](int r) {
        for (int k = 0; k < nseg; ++k)
            if (segbad[k] && r >= seg[5 * k + 3] && r < seg[5 * k + 4])
                return true;
        return false;
    };

    const int total = first[nseg];
    // Segment of a tile.  Each warp asks for its tiles in increasing order,
    // separately for issuing and for consuming, so each keeps a cursor that
    // only moves forward.
    auto seg_of = [&](int tile, int &k) {
        while (k + 1 < nseg && first[k + 1] <= tile)
            ++k;
        return k;
    };
    float *mw = reinterpret_cast<float *>(smem + C::OFF_STAGES);
    float *lw = mw + NW * RS;
    float *aw = lw + NW * RS;

    if (!invalid_item) {
        const int my_n = warp < total ? (total - 1 - warp) / NW + 1 : 0;
        uint8_t *stages = smem + C::OFF_STAGES + warp * S * C::STAGE_BYTES;
        uint64_t *bars = reinterpret_cast<uint64_t *>(smem + CC::OFF_BAR) + warp * S;
        int k_issue = 0, k_use = 0;
        auto issue = [&](int i, int st) {
            const int tile = warp + i * NW, k = seg_of(tile, k_issue);
            const int tb = seg[5 * k + 1], te = seg[5 * k + 2], j0 = tb / BS;
            const int t0 = tb + (tile - first[k]) * TILE;
            uint8_t *kd = stages + st * C::STAGE_BYTES;
            uint8_t *vd = kd + C::TILE_BYTES;
            const int nbox = min(C::BOXES, (te - t0 + C::BOX_ROWS - 1) / C::BOX_ROWS);
            mbar_arrive_expect_tx(&bars[st], (uint32_t)(nbox * 2 * C::BOX_BYTES));
            for (int b = 0; b < nbox; ++b) {
                const int tok = t0 + b * C::BOX_ROWS;
                const int phys = table_s[tab[k] + tok / BS - j0];
                tma_load_5d(kd + b * C::BOX_BYTES, &tmk, &bars[st], 0, tok % BS, 0, kvh, phys);
                tma_load_5d(vd + b * C::BOX_BYTES, &tmv, &bars[st], 0, tok % BS, 0, kvh, phys);
            }
        };
        if (lane == 0)
            for (int i = 0; i < (my_n < S ? my_n : S); ++i)
                issue(i, i);

        typename CC::Engine eng;
        eng.init(p, smem + CC::OFF_Q, w, warp, lane);
        int failed_at = -1;
        for (int i = 0; i < my_n; ++i) {
            const int st = i % S;
            if (!mbar_wait_bounded(&bars[st], (uint32_t)((i / S) & 1))) {
                failed_at = i;
                break;
            }
            const int tile = warp + i * NW, k = seg_of(tile, k_use);
            const int t0 = seg[5 * k + 1] + (tile - first[k]) * TILE;
            const int nvalid = min(TILE, seg[5 * k + 2] - t0);
            const uint32_t kbase = smem_u32(stages + st * C::STAGE_BYTES);
            eng.tile(kbase, kbase + C::TILE_BYTES, nvalid, lane, seg[5 * k + 3], seg[5 * k + 4]);
            __syncwarp();
            if (lane == 0 && i + S < my_n) {
                fence_proxy_async_smem();
                issue(i + S, st);
            }
        }
        if (failed_at >= 0) {
            const int last = min(my_n, failed_at + S);
            for (int i = failed_at; i < last; ++i)
                mbar_wait_bounded(&bars[i % S], (uint32_t)((i / S) & 1), 200000000ull);
            if (lane == 0) {
                report(p.status, PKV_DEV_TIMEOUT);
                atomicOr(cta_flag, 1u);
            }
        }
        __syncthreads();
        eng.finish(mw, lw, aw, warp, lane, nrows);
    }
    __syncthreads();

    // ---- this item's partial of every row (other CTAs read it through L2):
    // one thread per row folds the warps' (max, sum) and keeps the warps'
    // weights in shared memory; then float4 pieces of the accumulators.
    float *wts = reinterpret_cast<float *>(smem + CC::OFF_WTS);   // [RS][NW]
    const bool failed_all = invalid_item || *reinterpret_cast<volatile uint32_t *>(cta_flag) != 0;
    if (tid < nrows) {
        const int r = tid;
        const bool failed = failed_all || row_bad(r);
        float M = -INFINITY, den = 0.f, f[NW];
#pragma unroll
        for (int k = 0; k < NW; ++k)
            M = fmaxf(M, failed ? -INFINITY : mw[k * RS + r]);
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            const float mk = failed ? -INFINITY : mw[k * RS + r];
            f[k] = mk == -INFINITY ? 0.f : exp2f(mk - M);
            den += f[k] * lw[k * RS + r];
            wts[r * NW + k] = f[k];
        }
        const int64_t base = row_head(p, w, G, r) * slots + slot;
        __stcg(reinterpret_cast<float2 *>(p.ws_ml) + base,
               make_float2(failed ? -INFINITY : M, failed ? -1.f : den));
    }
    __syncthreads();
    for (int idx = tid; idx < nrows * (D / 4); idx += blockDim.x) {
        const int r = idx / (D / 4), d4 = idx % (D / 4);
        float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            const float f = wts[r * NW + k];
            const float4 a = reinterpret_cast<const float4 *>(aw + (k * RS + r) * D)[d4];
            num.x += f * a.x;
            num.y += f * a.y;
            num.z += f * a.z;
            num.w += f * a.w;
        }
        const int64_t base = row_head(p, w, G, r) * slots + slot;
        __stcg(reinterpret_cast<float4 *>(p.ws_acc + base * D) + d4, num);
    }

    // ---- arrivals: the CTA that delivers a sequence's last partial merges
    // it.  One thread per member: release this CTA's partials, count, and
    // acquire the others' before the merge reads them.
    __threadfence();
    __syncthreads();
    if (tid < nmem) {
        const int seq = seq0 + tid;
        int32_t *ctr = &counters[(int64_t)seq * Hk + kvh];
        __threadfence();
        const int old = atomicAdd(ctr, 1);
        const bool last = old == expected[seq] - 1;
        flag[tid] = last;
        if (last)
            *ctr = 0;  // every arrival is in: ready for the next call
        __threadfence();
    }
    __syncthreads();
    // the (member, head) rows of the completed members, spread over the warps
    int pr = 0;
    for (int m = 0; m < nmem; ++m) {
        if (!flag[m])
            continue;
        const int seq = seq0 + m;
        for (int h = 0; h < G; ++h, ++pr)
            if (pr % NW == warp)
                merge_partials<D>(p, (int64_t)seq * p.num_heads + kvh * G + h, expected[seq], slots,
                                  false, lane);
    }
}

}  // namespace pkv
