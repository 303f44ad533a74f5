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
//
// Latency is what this kernel fights (each CTA streams only a few hundred
// tokens): the item carries its physical block ids, so the first TMA loads
// leave one round trip after the CTA starts, and the check of the device
// block tables, the q staging and the merge bookkeeping run while they fly.
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
    static constexpr int TABLE_CAP = plan::kTableCap;
    // ring | barriers | flag | q rows | item copy (with its block ids) | first
    // tile / block-id offset / table-check offset / bad flag per segment,
    // merge flags, members' expected partial counts, bad-row and bad-length
    // masks | per-row warp weights
    static constexpr int OFF_STAGES = 0;
    static constexpr int OFF_BAR = C::STAGES_BYTES;
    static constexpr int OFF_FLAG = OFF_BAR + NW * S * 8;
    static constexpr int OFF_Q = OFF_FLAG + 16;
    static constexpr int OFF_ITEM = OFF_Q + Engine::q_smem_bytes;
    static constexpr int EXTRA_INTS = ITEM_INTS + 4 * (MAXSEG + 1) + 2 * plan::kMaxRows + 2;
    static constexpr int OFF_WTS = (OFF_ITEM + EXTRA_INTS * 4 + 15) / 16 * 16;
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
    constexpr int AWS = CC::Engine::AWS;
    static_assert(NW * RS * (AWS + 2) * 4 <= C::STAGES_BYTES, "merge scratch fits in the ring");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = aligned_smem(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kvh = blockIdx.x, item = blockIdx.y;

    // plan geometry from the launch: B and Hk fix where the items start,
    // the slot count is the workspace's row stride
    const int B = p.num_seqs, Hk = p.num_kv_heads, slots = p.num_partitions;
    const int32_t *expected = plan_buf + plan::kHeader;
    const int32_t *plan_lens = expected + B;
    int32_t *counters = plan_buf + plan::kHeader + 2 * B;
    const int32_t *src = counters + (int64_t)B * Hk + (int64_t)item * CC::ITEM_INTS;

    int32_t *it = reinterpret_cast<int32_t *>(smem + CC::OFF_ITEM);
    int32_t *first = it + CC::ITEM_INTS;     // first tile of segment k (k <= nseg)
    int32_t *tab = first + CC::MAXSEG + 1;   // offset of segment k's block ids
    int32_t *vtab = tab + CC::MAXSEG + 1;    // first table check of segment k
    int32_t *segbad = vtab + CC::MAXSEG + 1; // segment k addresses a bad block
    int32_t *flag = segbad + CC::MAXSEG + 1; // merge flags per member
    int32_t *exp_s = flag + plan::kMaxRows;  // expected partials per member
    uint32_t *badrows = reinterpret_cast<uint32_t *>(exp_s + plan::kMaxRows);
    uint32_t *lenbad = badrows + 1;          // members whose device length differs from the plan's
    uint32_t *cta_flag = reinterpret_cast<uint32_t *>(smem + CC::OFF_FLAG);
    {
        // all loads in flight before the first store (see stage_q_rows)
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
    init_rings<CC>(smem);
    if (tid == 0) {
        *cta_flag = 0;
        *lenbad = 0;
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
    }
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
    int32_t *ids = it + CC::IDS;             // the segments' physical block ids
    // a segment that covers every row of a multi-member item is a shared
    // prefix: every member's table must hold its block ids
    auto shared_seg = [&](int k) {
        return seg[5 * k + 3] == 0 && seg[5 * k + 4] == nrows && nmem > 1;
    };
    if (tid == 0) {
        int tiles = 0, entries = 0, checks = 0;
        for (int k = 0; k < nseg; ++k) {
            first[k] = tiles;
            tab[k] = entries;
            vtab[k] = checks;
            segbad[k] = 0;
            const int b = seg[5 * k + 1], e = seg[5 * k + 2];
            const int nb = (e + BS - 1) / BS - b / BS;
            tiles += (e - b + TILE - 1) / TILE;
            entries += nb;
            checks += (shared_seg(k) ? nmem : 1) * nb;
        }
        first[nseg] = tiles;
        tab[nseg] = entries;
        vtab[nseg] = checks;
    }
    __syncthreads();

    // ---- block ids outside the pool invalidate their segment's rows (block
    // 0 is loaded in their place); this must precede the first load
    const bool invalid_item = tab[nseg] > CC::TABLE_CAP;
    if (!invalid_item)
        for (int k = 0; k < nseg; ++k)
            for (int i = tab[k] + tid; i < tab[k + 1]; i += blockDim.x) {
                const int b = ids[i];
                if (b < 0 || (int64_t)b >= p.num_blocks) {
                    segbad[k] = 1;
                    ids[i] = 0;
                }
            }
    __syncthreads();

    const int total = first[nseg];
    // Segment of a tile.  Each warp asks for its tiles in increasing order,
    // separately for issuing and for consuming, so each keeps a cursor that
    // only moves forward.
    auto seg_of = [&](int tile, int &k) {
        while (k + 1 < nseg && first[k + 1] <= tile)
            ++k;
        return k;
    };
    const int my_n = invalid_item ? 0 : (warp < total ? (total - 1 - warp) / NW + 1 : 0);
    uint8_t *stages = smem + CC::OFF_STAGES + warp * S * C::STAGE_BYTES;
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
            const int phys = ids[tab[k] + tok / BS - j0];
            tma_load_5d(kd + b * C::BOX_BYTES, &tmk, &bars[st], 0, tok % BS, 0, kvh, phys);
            tma_load_5d(vd + b * C::BOX_BYTES, &tmv, &bars[st], 0, tok % BS, 0, kvh, phys);
        }
    };
    if (lane == 0)
        for (int i = 0; i < (my_n < S ? my_n : S); ++i)
            issue(i, i);

    // ---- while the first tiles load: the device tables must hold the plan's
    // block ids (every member's table for a shared prefix segment, the
    // segment's own table otherwise); q rows to shared memory; the members'
    // expected partial counts.  Table entries are checked four per thread at
    // a time, loads first.
    if (!invalid_item) {
        const int vtotal = vtab[nseg];
        for (int x0 = 0; x0 < vtotal; x0 += 4 * NW * 32) {
            int got[4], want[4], kk[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int x = x0 + u * NW * 32 + tid;
                kk[u] = -1;
                got[u] = want[u] = 0;
                if (x < vtotal) {
                    int k = 0;
                    while (k + 1 < nseg && vtab[k + 1] <= x)
                        ++k;
                    const int nb = tab[k + 1] - tab[k], local = x - vtab[k];
                    const int m = local / nb, i = local % nb;
                    const int s = shared_seg(k) ? seq0 + m : seg[5 * k];
                    got[u] = p.block_tables[(int64_t)s * p.max_blocks_per_seq + seg[5 * k + 1] / BS + i];
                    want[u] = ids[tab[k] + i];
                    kk[u] = k;
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (kk[u] >= 0 && got[u] != want[u])
                    segbad[kk[u]] = 1;
        }
    }
    CC::Engine::stage_q_rows(p, smem + CC::OFF_Q, w);
    if (tid < nmem) {
        exp_s[tid] = expected[seq0 + tid];
        if (plan_lens[seq0 + tid] != p.context_lens[seq0 + tid])
            atomicOr(lenbad, 1u << tid);
    }
    __syncthreads();
    if (tid == 0) {
        bool any = invalid_item;
        uint32_t mask = 0;
        for (int k = 0; k < nseg; ++k)
            if (segbad[k]) {
                any = true;
                for (int r = seg[5 * k + 3]; r < seg[5 * k + 4]; ++r)
                    mask |= 1u << r;
            }
        const uint32_t lb = *lenbad;
        for (int m = 0; m < nmem; ++m)
            if ((lb >> m) & 1u)
                mask |= ((1u << G) - 1u) << (m * G);
        *badrows = mask;
        if (any)
            report(p.status, PKV_DEV_BAD_BLOCK);
        if (lb)
            report(p.status, PKV_DEV_BAD_CONTEXT_LEN);
    }

    float *mw = reinterpret_cast<float *>(smem + C::OFF_STAGES);
    float *lw = mw + NW * RS;
    float *aw = lw + NW * RS;
    if (!invalid_item) {
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

    // ---- every row's result: the output itself for a sequence this item
    // holds entirely, otherwise this item's partial (read by other CTAs
    // through L2).  One thread per row folds the warps' (max, sum) into
    // weights in shared memory (1 / sum included for a final row); then float4
    // pieces of the accumulators.
    float *wts = reinterpret_cast<float *>(smem + CC::OFF_WTS);   // [RS][NW]
    const bool failed_all = invalid_item || *reinterpret_cast<volatile uint32_t *>(cta_flag) != 0;
    if (tid < nrows) {
        const int r = tid;
        const bool failed = failed_all || ((*badrows >> r) & 1u);
        const bool final_row = exp_s[r / G] == 1;
        float M = -INFINITY, den = 0.f, f[NW];
#pragma unroll
        for (int k = 0; k < NW; ++k)
            M = fmaxf(M, failed ? -INFINITY : mw[k * RS + r]);
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            const float mk = failed ? -INFINITY : mw[k * RS + r];
            f[k] = mk == -INFINITY ? 0.f : exp2f(mk - M);
            den += f[k] * lw[k * RS + r];
        }
        const float norm = !final_row ? 1.f : (den > 0.f ? 1.f / den : 0.f);
#pragma unroll
        for (int k = 0; k < NW; ++k)
            wts[r * NW + k] = f[k] * norm;
        if (!final_row) {
            const int64_t base = row_head(p, w, G, r) * slots + slot;
            __stcg(reinterpret_cast<float2 *>(p.ws_ml) + base,
                   make_float2(failed ? -INFINITY : M, failed ? -1.f : den));
        }
    }
    __syncthreads();
    for (int idx = tid; idx < nrows * (D / 4); idx += blockDim.x) {
        const int r = idx / (D / 4), d4 = idx % (D / 4);
        float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            const float f = wts[r * NW + k];
            const float4 a = reinterpret_cast<const float4 *>(aw + (k * RS + r) * AWS)[d4];
            num.x += f * a.x;
            num.y += f * a.y;
            num.z += f * a.z;
            num.w += f * a.w;
        }
        const int64_t sh = row_head(p, w, G, r);
        if (exp_s[r / G] == 1) {
            const int64_t o = sh * D + 4 * d4;
            store_out(p.out, p.out_dtype, o + 0, num.x);
            store_out(p.out, p.out_dtype, o + 1, num.y);
            store_out(p.out, p.out_dtype, o + 2, num.z);
            store_out(p.out, p.out_dtype, o + 3, num.w);
        } else {
            __stcg(reinterpret_cast<float4 *>(p.ws_acc + (sh * slots + slot) * D) + d4, num);
        }
    }

    // ---- arrivals: the CTA that delivers a sequence's last partial merges
    // it.  After the barrier, one thread per member releases the CTA's
    // partials (fence, then count) and, if its count completes the sequence,
    // acquires the other CTAs' partials (fence) before the barrier that
    // precedes the merge reads.
    __syncthreads();
    if (tid < nmem) {
        flag[tid] = 0;
        if (exp_s[tid] > 1) {   // a sequence held by this item alone is done
            int32_t *ctr = &counters[(int64_t)(seq0 + tid) * Hk + kvh];
            __threadfence();
            const int old = atomicAdd(ctr, 1);
            const bool last = old == exp_s[tid] - 1;
            flag[tid] = last;
            if (last) {
                *ctr = 0;  // every arrival is in: ready for the next call
                __threadfence();
            }
        }
    }
    __syncthreads();
    // the (member, head) rows of the completed members, one half-warp each
    const int hw = tid >> 4, hl = tid & 15;
    int pr = 0;
    for (int m = 0; m < nmem; ++m) {
        if (!flag[m])
            continue;
        const int seq = seq0 + m;
        for (int h = 0; h < G; ++h, ++pr)
            if (pr % (2 * NW) == hw)
                merge_partials<D>(p, (int64_t)seq * p.num_heads + kvh * G + h, exp_s[m], slots,
                                  false, hl);
    }
}

}  // namespace pkv
