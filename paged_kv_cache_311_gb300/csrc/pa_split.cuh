// pa_split.cuh -- persistent split-context decode (16-bit caches, tensor-core
// engine) and the log-sum-exp merge of its partials.
//
// Work is cut into items; an item is one partition of at most P tokens of one
// kv head, for up to 8 query rows (the G heads of one sequence, or 8 rows of
// the heads of several sequences that share the partition's blocks).  Every
// warp of the grid is an independent worker that walks the items gw, gw + W,
// gw + 2W, ... (W warps in the grid).  Lane 0 of the warp runs the TMA
// producer S tiles ahead of the warp's own consumption, straight across item
// boundaries, so the pipeline never drains between items; the partition's
// slice of the block table is staged into the warp's shared memory when the
// producer reaches the item.  Each finished item writes its partial (max,
// sum, unnormalised acc per row) to its workspace slot; pa_merge_kernel then
// merges the slots of every (sequence, head) with log-sum-exp weights.
//
// Item sources: the plain split path enumerates (sequence, kv head,
// partition) implicitly; the shared-prefix path reads an explicit item list
// that pa_plan_kernel builds (pa_shared.cuh).
#pragma once

#include "pa_decode.cuh"

namespace pkv {

struct SplitItem {
    int seq0;        // first sequence of the item's rows
    int nrows;       // live query rows (<= 8 per row block, G per sequence)
    int kvh;
    int rb;          // row block: rows 8 rb .. 8 rb + 7
    int tok_begin;   // token range of the item (multiple of the tile)
    int tok_end;
    int slot;        // workspace slot of every row's (sequence, head)
    int table_seq;   // sequence whose block table addresses the tokens
};

// Explicit items are stored as two int4: {seq0, nrows, kvh, rb}, {tok_begin,
// tok_end, slot, table_seq}.
__device__ __forceinline__ SplitItem load_item(const int4 *items, int idx)
{
    const int4 a = items[2 * idx], b = items[2 * idx + 1];
    return SplitItem{a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
}

template <typename T, int D, int BS, int G>
struct SplitCfg {
    using C = DecodeCfg<T, D, BS, G, true>;
    static constexpr int NW = 4;
    static constexpr int S = C::S;
    static constexpr int TABLE_W = 128;             // block-table entries per warp
    static constexpr int OFF_STAGES = 0;
    static constexpr int OFF_TABLE = NW * S * C::STAGE_BYTES;
    static constexpr int OFF_META = OFF_TABLE + NW * TABLE_W * 4;
    static constexpr int OFF_BAR = OFF_META + NW * S * 32;
    static constexpr int SMEM_BYTES = OFF_BAR + NW * S * 8 + 1024;
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

template <typename T, int D, int BS, int G, bool EXPLICIT>
__global__ void __launch_bounds__(128)
pa_split_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                const __grid_constant__ CUtensorMap tmv)
{
    using SC = SplitCfg<T, D, BS, G>;
    using C = typename SC::C;
    constexpr int S = SC::S, TILE = C::TILE;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gw = blockIdx.x * SC::NW + warp;
    const int W = gridDim.x * SC::NW;

    uint8_t *stages = smem + SC::OFF_STAGES + warp * S * C::STAGE_BYTES;
    int32_t *tbl = reinterpret_cast<int32_t *>(smem + SC::OFF_TABLE) + warp * SC::TABLE_W;
    int4 *meta = reinterpret_cast<int4 *>(smem + SC::OFF_META) + warp * S * 2;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SC::OFF_BAR) + warp * S;
    if (lane == 0) {
        for (int s = 0; s < S; ++s)
            mbar_init(&bars[s], 1);
        fence_mbar_init();
        if (warp == 0) {
            prefetch_tensormap(&tmk);
            prefetch_tensormap(&tmv);
        }
    }
    __syncwarp();

    const int np = p.num_partitions;
    const long long total = EXPLICIT ? (long long)*p.num_items
                                     : (long long)p.num_seqs * p.num_kv_heads * np;

    // ---------------------------------------------------------- producer
    long long p_idx = (long long)gw - W;
    SplitItem pit{};
    int p_tile = 0, p_ntiles = 0, p_st = 0, p_j0 = 0, p_bad = 0;
    bool p_done = false, p_sent = false;

    auto fetch = [&](long long idx, SplitItem &it) {
        if constexpr (EXPLICIT) {
            it = load_item(p.items, (int)idx);
        } else {
            const int part = (int)(idx % np);
            const long long sk = idx / np;
            const int kvh = (int)(sk % p.num_kv_heads), seq = (int)(sk / p.num_kv_heads);
            const int L = p.context_lens[seq];
            it.seq0 = seq;
            it.nrows = G;
            it.kvh = kvh;
            it.rb = 0;
            it.tok_begin = part * p.partition_size;
            // a bad length leaves the item empty: the merge kernel zeroes the row
            it.tok_end = (L < 0 || L > p.max_context_len) ? 0 : min(it.tok_begin + p.partition_size, L);
            it.slot = part;
            it.table_seq = seq;
        }
    };

    // Whole warp: issues the next tile (or the end-of-work sentinel) into the
    // stage p_st.
    auto produce = [&]() {
        if (p_sent)
            return;
        if (!p_done && p_tile == p_ntiles) {
            for (;;) {
                p_idx += W;
                if (p_idx >= total) {
                    p_done = true;
                    break;
                }
                fetch(p_idx, pit);
                if (pit.tok_end > pit.tok_begin)
                    break;
            }
            if (!p_done) {
                p_j0 = pit.tok_begin / BS;
                const int nb = (pit.tok_end - pit.tok_begin + BS - 1) / BS;
                const int32_t *bt = p.block_tables + (int64_t)pit.table_seq * p.max_blocks_per_seq + p_j0;
                int bad = 0;
                for (int j = lane; j < nb; j += 32) {
                    int b = bt[j];
                    if (b < 0 || (int64_t)b >= p.num_blocks) {
                        bad = 1;
                        b = 0;
                    }
                    tbl[j] = b;
                }
                p_bad = __any_sync(0xffffffffu, bad);
                __syncwarp();
                p_tile = 0;
                p_ntiles = (pit.tok_end - pit.tok_begin + TILE - 1) / TILE;
            }
        }
        if (lane == 0) {
            int4 *mt = meta + 2 * p_st;
            if (p_done) {
                mt[0] = make_int4(-1, 0, 0, 0);
                mbar_arrive(&bars[p_st]);
            } else {
                const int t0 = pit.tok_begin + p_tile * TILE;
                const int nvalid = min(TILE, pit.tok_end - t0);
                const int flags = (p_tile == 0 ? 1 : 0) | (p_tile == p_ntiles - 1 ? 2 : 0) | (p_bad ? 4 : 0);
                mt[0] = make_int4(pit.seq0, pit.nrows, pit.kvh, pit.rb);
                mt[1] = make_int4(pit.slot, nvalid, flags, 0);
                uint8_t *kd = stages + p_st * C::STAGE_BYTES;
                uint8_t *vd = kd + C::TILE_BYTES;
                const int nbox = (nvalid + C::BOX_ROWS - 1) / C::BOX_ROWS;
                mbar_arrive_expect_tx(&bars[p_st], (uint32_t)(nbox * 2 * C::BOX_BYTES));
                for (int b = 0; b < nbox; ++b) {
                    const int tok = t0 + b * C::BOX_ROWS;
                    const int phys = tbl[tok / BS - p_j0];
                    const int row0 = tok % BS;
                    tma_load_5d(kd + b * C::BOX_BYTES, &tmk, &bars[p_st], 0, row0, 0, pit.kvh, phys);
                    tma_load_5d(vd + b * C::BOX_BYTES, &tmv, &bars[p_st], 0, row0, 0, pit.kvh, phys);
                }
            }
        }
        if (p_done)
            p_sent = true;
        else
            ++p_tile;
        p_st = p_st + 1 == S ? 0 : p_st + 1;
    };

    for (int i = 0; i < S; ++i)
        produce();

    // ---------------------------------------------------------- consumer
    TcEngine<T, D, BS, G> eng;
    int c_st = 0;
    for (long long n = 0;; ++n) {
        if (!mbar_wait_bounded(&bars[c_st], (uint32_t)((n / S) & 1))) {
            // Give up: wait (bounded) for the stages still in flight, report.
            for (int k = 1; k < S; ++k) {
                const long long m = n + k;
                mbar_wait_bounded(&bars[m % S], (uint32_t)((m / S) & 1), 200000000ull);
            }
            if (lane == 0)
                report(p.status, PKV_DEV_TIMEOUT);
            return;
        }
        const int4 m0 = meta[2 * c_st], m1 = meta[2 * c_st + 1];
        if (m0.x < 0)
            break;  // sentinel: no more work for this warp
        const int seq0 = m0.x, nrows = m0.y, kvh = m0.z, rb = m0.w;
        const int slot = m1.x, nvalid = m1.y, flags = m1.z;
        if (flags & 1)
            eng.begin_item(p, seq0, nrows, kvh, rb, lane);
        const uint32_t kbase = smem_u32(stages + c_st * C::STAGE_BYTES);
        eng.tile(kbase, kbase + C::TILE_BYTES, nvalid, lane);
        if (flags & 2) {
            eng.write_partial(p, seq0, nrows, kvh, rb, slot, (flags & 4) != 0);
            if ((flags & 4) && lane == 0)
                report(p.status, PKV_DEV_BAD_BLOCK);
        }
        __syncwarp();
        if (lane == 0)
            fence_proxy_async_smem();  // our reads of the stage precede its next TMA write
        produce();
        c_st = c_st + 1 == S ? 0 : c_st + 1;
    }
}

// Log-sum-exp merge of the partials of one (sequence, head) per CTA.  The
// valid slots are [0, ceil(S / P)) for a shared prefix of S tokens (only in
// the shared-prefix path) and [np_prefix, np_prefix + ceil((L - S) / P)).
template <int D>
__global__ void __launch_bounds__(128) pa_merge_kernel(const __grid_constant__ DecodeParams p)
{
    constexpr int DPL = D / 32;
    __shared__ float red_m[4];
    __shared__ int red_bad[4];
    __shared__ float part_num[4][D];
    __shared__ float part_den[4];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t sh = blockIdx.x;
    const int seq = (int)(sh / p.num_heads);
    const int L = p.context_lens[seq];
    const bool bad_len = L < 0 || L > p.max_context_len;
    if (bad_len && threadIdx.x == 0 && sh % p.num_heads == 0)
        report(p.status, PKV_DEV_BAD_CONTEXT_LEN);  // the item pass skipped it silently
    const int S = (!bad_len && p.seq_shared) ? p.seq_shared[seq] : 0;
    const int P = p.partition_size;
    const int na = S > 0 ? (S + P - 1) / P : 0;
    const int nb = bad_len ? 0 : (L - S + P - 1) / P;
    const int n = na + nb;
    auto slot_of = [&](int k) { return k < na ? k : p.np_prefix + (k - na); };
    const float *ml = p.ws_ml + sh * p.num_partitions * 2;
    const float *accp = p.ws_acc + sh * p.num_partitions * D;

    float M = -INFINITY;
    int invalid = 0;
    for (int k = threadIdx.x; k < n; k += blockDim.x) {
        const int sl = slot_of(k);
        M = fmaxf(M, ml[2 * sl]);
        invalid |= ml[2 * sl + 1] < 0.f;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    invalid = __any_sync(0xffffffffu, invalid);
    if (lane == 0) {
        red_m[warp] = M;
        red_bad[warp] = invalid;
    }
    __syncthreads();
    M = fmaxf(fmaxf(red_m[0], red_m[1]), fmaxf(red_m[2], red_m[3]));
    invalid = red_bad[0] | red_bad[1] | red_bad[2] | red_bad[3];

    float num[DPL];
#pragma unroll
    for (int k = 0; k < DPL; ++k)
        num[k] = 0.f;
    float den = 0.f;
    if (!invalid && !bad_len) {
        // warp w takes slots w, w + 4, ...; two loads in flight per lane
        for (int k = warp; k < n; k += 8) {
            const int k2 = k + 4;
            const int s1 = slot_of(k);
            const float m1 = ml[2 * s1], l1 = ml[2 * s1 + 1];
            const float *a1 = accp + (int64_t)s1 * D + lane * DPL;
            float v1[DPL], v2[DPL];
            float m2 = -INFINITY, l2 = 0.f;
            if constexpr (DPL == 4) {
                const float4 t = *reinterpret_cast<const float4 *>(a1);
                v1[0] = t.x; v1[1] = t.y; v1[2] = t.z; v1[3] = t.w;
            } else {
                const float2 t = *reinterpret_cast<const float2 *>(a1);
                v1[0] = t.x; v1[1] = t.y;
            }
            if (k2 < n) {
                const int s2 = slot_of(k2);
                m2 = ml[2 * s2];
                l2 = ml[2 * s2 + 1];
                const float *a2 = accp + (int64_t)s2 * D + lane * DPL;
                if constexpr (DPL == 4) {
                    const float4 t = *reinterpret_cast<const float4 *>(a2);
                    v2[0] = t.x; v2[1] = t.y; v2[2] = t.z; v2[3] = t.w;
                } else {
                    const float2 t = *reinterpret_cast<const float2 *>(a2);
                    v2[0] = t.x; v2[1] = t.y;
                }
            }
            if (m1 != -INFINITY) {
                const float f = exp2f(m1 - M);
                den += f * l1;
#pragma unroll
                for (int d = 0; d < DPL; ++d)
                    num[d] += f * v1[d];
            }
            if (m2 != -INFINITY) {
                const float f = exp2f(m2 - M);
                den += f * l2;
#pragma unroll
                for (int d = 0; d < DPL; ++d)
                    num[d] += f * v2[d];
            }
        }
    }
#pragma unroll
    for (int d = 0; d < DPL; ++d)
        part_num[warp][lane * DPL + d] = num[d];
    if (lane == 0)
        part_den[warp] = den;
    __syncthreads();
    const float dsum = part_den[0] + part_den[1] + part_den[2] + part_den[3];
    const bool zero = invalid || bad_len || dsum == 0.f;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        const float v = part_num[0][d] + part_num[1][d] + part_num[2][d] + part_num[3][d];
        store_out(p.out, p.out_dtype, sh * D + d, zero ? 0.f : v / dsum);
    }
}

}  // namespace pkv
