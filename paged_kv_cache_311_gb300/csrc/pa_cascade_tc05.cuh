// pa_cascade_tc05.cuh -- shared-prefix (cascade) decode on the 5th-generation
// tensor cores (tcgen05).
//
// Same plan, items, device checks and partials as pa_cascade_kernel
// (cascade_plan.h; PagedAttention: Efficient LLM Serving with vLLM,
// "Advanced Features", KV-Cache Sharing), with the attention products moved
// from per-warp mma.sync to tcgen05.mma issued by one thread, accumulators in
// tensor memory (TMEM):
//   * A CTA-wide ring of four 32-token stages (two 16-token tiles each): per
//     stage K and V, each as two planes [64-element chunk][32 rows][128 B]
//     with 128-byte swizzling, written by one TMA load per block box and
//     chunk.
//   * S^T = K q^T: M = 64 tokens (the stage's 32 and 32 ignored rows), N = 8
//     x the item's n-tiles of query rows, K = head_dim, into TMEM columns
//     [0, 24); row r of S^T sits in TMEM lane 32 (r / 16) + r % 16, so warps
//     0 and 1 read the scores of their tile's 16 tokens from their own lane
//     quarters.
//   * Online softmax in the log2 domain against a CTA-wide reference maximum
//     per query row, kept while every new score stays within kSlack of it;
//     otherwise the CTA moves to the exact running maxima and rescales O in
//     TMEM.  P (<= 2^kSlack) is split into a 16-bit high part and remainder,
//     written over the stage's K (no longer needed) as [query row][token].
//   * O^T += V^T P^T: M = 128 dims (V read MN-major), N = query rows, K = 16
//     tokens per instruction, high and low parts into the same accumulator
//     (TMEM columns [32, 56)); its completion frees the stage for the TMA.
//   * End of an item: O^T read from TMEM (thread = one dim, registers = rows),
//     row sums reduced across the tokens' lanes, output or partial written.
#pragma once

#include "pa_cascade.cuh"

namespace pkv {

// fp32 -> the cache's 16-bit type, round to nearest even
template <typename T> __device__ __forceinline__ T to_elem(float v);
template <> __device__ __forceinline__ __nv_bfloat16 to_elem<__nv_bfloat16>(float v)
{
    return __float2bfloat16_rn(v);
}
template <> __device__ __forceinline__ __half to_elem<__half>(float v) { return __float2half_rn(v); }

template <typename T, int D, int BS, int G>
struct Tc05Cfg {
    static_assert(D == 128, "the tcgen05 cascade kernel takes head_dim 128");
    static constexpr int NW = 4;
    static constexpr int TILE = plan::kTileTokens;   // 16 tokens
    static constexpr int TOK = 2 * TILE;             // tokens per stage
    static constexpr int GRP = 8;                    // tokens per group: one 8-row swizzle atom
    static constexpr int NSLOT = 4;                  // stages in the ring
    static constexpr int CHUNKS = D * 2 / 128;       // 64-element chunks per row
    static constexpr int ATOM = GRP * 128;           // one chunk of one group's rows
    // a group's period: [K chunk 0][K chunk 1][V chunk 0][V chunk 1]
    static constexpr int PERIOD = 4 * ATOM;
    static constexpr int V_OFF = 2 * ATOM;
    static constexpr int SLOT = (TOK / GRP) * PERIOD;
    static constexpr int BOX_ROWS = GRP;
    static constexpr int RQ = plan::kMaxRows;        // query rows of an item
    static constexpr int RPL = RQ / 4;               // query rows per lane (four lanes per token)
    static constexpr int QPLANE = RQ * 128;
    static constexpr int TM_COLS = 64;               // S^T at column 0, O^T at column 32
    static constexpr int MAXSEG = plan::max_segments(G);
    static constexpr int ITEM_INTS = plan::item_ints(G);
    static constexpr int IDS = plan::item_ids_offset(G);
    static constexpr int SEGS = plan::item_segments_offset();
    static constexpr int TABLE_CAP = plan::kTableCap;
    // ring | q rows | barriers (full[NSLOT], empty[NSLOT], scores) | TMEM
    // address, flag, stages issued | per-warp row reductions [NW][RQ], the
    // rows' reference maxima and rescale factors | item copy, segment /
    // member / row flags | the list's next item
    static constexpr int OFF_RING = 0;
    static constexpr int OFF_Q = NSLOT * SLOT;
    static constexpr int OFF_BAR = OFF_Q + CHUNKS * QPLANE;
    static constexpr int OFF_TMEM = OFF_BAR + (2 * NSLOT + 1) * 8;
    static constexpr int OFF_FLAG = OFF_TMEM + 8;
    static constexpr int OFF_RED = OFF_FLAG + 8;
    static constexpr int OFF_ITEM = (OFF_RED + (NW + 2) * RQ * 4 + 15) / 16 * 16;
    static constexpr int EXTRA_INTS = ITEM_INTS + MAXSEG + RQ + 2;
    static constexpr int OFF_NEXT = (OFF_ITEM + EXTRA_INTS * 4 + 15) / 16 * 16;
    static constexpr bool PREFETCH = 3 * (OFF_NEXT + ITEM_INTS * 4 + 2048) <= 228 * 1024;
    static constexpr int SMEM_USED = OFF_NEXT + (PREFETCH ? ITEM_INTS * 4 : 0);
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;   // slack for 1024-byte alignment
    static_assert(3 * (SMEM_BYTES + 1024) <= 228 * 1024, "three CTAs per SM");
    static_assert(3 * TM_COLS <= 512, "TMEM of three CTAs per SM");
    static_assert(SLOT % 1024 == 0 && OFF_Q % 1024 == 0 && QPLANE % 1024 == 0 && ATOM == 1024,
                  "128-byte swizzle atoms are 1024-byte aligned");
    // S^T's A operand spans 16 atoms from a slot's chunk-1 start: the last
    // one reads the 1 KiB after the slot (the next slot, or the q rows); an
    // M = 128 product's N rounded up to 32 reads q rows 24-31 past the staged
    // ones (in shared memory; their columns are never read)
    static_assert(OFF_Q >= SLOT && CHUNKS == 2 && TOK / GRP == NW, "layout");
    static_assert(plan::kNT * 8 == RQ && RQ % 4 == 0 && (RPL % 2) == 0, "n-tiles");
};

template <typename T, int D, int BS, int G>
__global__ void __launch_bounds__(128, 3)
pa_cascade_tc05_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv, const int32_t *plan_buf)
{
    using CC = Tc05Cfg<T, D, BS, G>;
    constexpr int NW = CC::NW, TILE = CC::TILE, NSLOT = CC::NSLOT, RQ = CC::RQ, NT = plan::kNT;
    constexpr float kSlack = 8.f;
    constexpr int kIssuer = 64;     // lane 0 of warp 2: issues the MMAs
    constexpr int kProducer = 96;   // lane 0 of warp 3: issues the TMA loads
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = aligned_smem(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kvh = blockIdx.x;

    uint64_t *full = reinterpret_cast<uint64_t *>(smem + CC::OFF_BAR);
    uint64_t *empty = full + NSLOT;
    uint64_t *sbar = empty + NSLOT;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + CC::OFF_TMEM);
    uint32_t *cta_flag = reinterpret_cast<uint32_t *>(smem + CC::OFF_FLAG);
    int32_t *n_issued = reinterpret_cast<int32_t *>(cta_flag + 1);   // stages of the item issued
    float *red = reinterpret_cast<float *>(smem + CC::OFF_RED);   // [NW][RQ]
    float *mref = red + NW * RQ;  // the rows' reference maxima (log2 domain), CTA-uniform
    float *alph = mref + RQ;      // rescale factors of a moved reference
    int32_t *it = reinterpret_cast<int32_t *>(smem + CC::OFF_ITEM);
    int32_t *segbad = it + CC::ITEM_INTS;
    int32_t *exp_s = segbad + CC::MAXSEG;
    uint32_t *badrows = reinterpret_cast<uint32_t *>(exp_s + RQ);
    uint32_t *lenbad = badrows + 1;
    int32_t *next_buf = reinterpret_cast<int32_t *>(smem + CC::OFF_NEXT);
    const uint32_t qb = smem_u32(smem + CC::OFF_Q);

    const int B = p.num_seqs, slots = p.num_partitions;
    const int32_t *expected = plan_buf + plan::kHeader;
    const int32_t *plan_lens = expected + B;
    const int32_t *items = plan_buf + plan::kHeader + 2 * B;

    if (tid == 0) {
        for (int i = 0; i < 2 * NSLOT + 1; ++i)
            mbar_init(&full[i], 1);
        fence_mbar_init();
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
        *cta_flag = 0;
    }
    if (warp == 0)
        tc05::alloc(tslot, CC::TM_COLS);
    tc05::fence_before_sync();
    __syncthreads();
    tc05::fence_after_sync();
    const uint32_t tS = *tslot, tO = tS + 32;
    const uint32_t tlane = (uint32_t)(32 * warp) << 16;   // this warp's lane quarter
    // launched as a programmatic dependent of the previous kernel: nothing it
    // may write is read before this wait; only then may the merge kernel
    // behind this grid start (it reads the plan before its own wait)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    int g = 0;   // stages this CTA has started, over all its items
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
        const int32_t *members = it + plan::kItemHead;
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
        auto seg = [&](int k) { return it + CC::SEGS + plan::kSegInts * k; };
        int32_t *ids = it + CC::IDS;
        const bool dead = *reinterpret_cast<volatile uint32_t *>(cta_flag) != 0;
        const bool invalid_item =
            it[plan::I_IDS] > CC::TABLE_CAP || nseg > CC::MAXSEG || nrows > RQ || nrows <= 0;
        auto seg_of = [&](int tile, int &k) {
            while (k + 1 < nseg && seg(k + 1)[plan::S_FIRST_TILE] <= tile)
                ++k;
            return k;
        };
        const int n_st = invalid_item || dead ? 0 : (total + 1) / 2;
        const int ntl = (nrows + 7) / 8;
        int k_issue = 0;
        // Stage s of the item (its tiles 2s, 2s + 1) into the ring slot of
        // CTA stage g + s: one TMA load per block box, chunk plane and
        // matrix.  A block id outside the pool invalidates its segment's rows
        // (block 0 is loaded in its place).
        auto issue = [&](int s) {
            const int gs = g + s, sl = gs % NSLOT;
            uint8_t *base = smem + CC::OFF_RING + sl * CC::SLOT;
            int kk[2], t0[2], te[2];
            uint32_t bytes = 0;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int tt = 2 * s + u;
                te[u] = 0;
                t0[u] = 0;
                if (tt < total) {
                    kk[u] = seg_of(tt, k_issue);
                    const int *gg = seg(kk[u]);
                    t0[u] = gg[plan::S_BEGIN] + (tt - gg[plan::S_FIRST_TILE]) * TILE;
                    te[u] = min(gg[plan::S_END], t0[u] + TILE);
                    bytes += (uint32_t)(((te[u] - t0[u] + CC::GRP - 1) / CC::GRP) * 4 * CC::ATOM);
                }
            }
            mbar_arrive_expect_tx(&full[sl], bytes);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                for (int gi = 0; gi < 2; ++gi) {
                    const int tok = t0[u] + gi * CC::GRP;
                    if (tok >= te[u])
                        continue;
                    const int *gg = seg(kk[u]);
                    int phys = ids[gg[plan::S_ID_OFF] + tok / BS - gg[plan::S_BEGIN] / BS];
                    if (phys < 0 || (int64_t)phys >= p.num_blocks) {
                        segbad[kk[u]] = 1;
                        phys = 0;
                    }
                    uint8_t *gb = base + (2 * u + gi) * CC::PERIOD;
#pragma unroll
                    for (int c = 0; c < CC::CHUNKS; ++c) {
                        tma_load_5d(gb + c * CC::ATOM, &tmk, &full[sl], 0, tok % BS, c, kvh, phys);
                        tma_load_5d(gb + CC::V_OFF + c * CC::ATOM, &tmv, &full[sl], 0, tok % BS, c, kvh, phys);
                    }
                }
            }
        };
        if (tid == kProducer) {
            *n_issued = min(n_st, NSLOT - 1);
            for (int s = 0; s < min(n_st, NSLOT - 1); ++s)
                issue(s);
        }

        // ---- while the first stages load, one round trip of global loads:
        // the device table entries to check against the plan's block ids,
        // the q rows and the members' expected partial counts and lengths
        const int vtotal = invalid_item ? 0 : it[plan::I_CHECKS];
        int got[4], want[4], kk4[4];
        auto load_checks = [&](int x0) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int x = x0 + u * NW * 32 + tid;
                kk4[u] = -1;
                got[u] = want[u] = 0;
                if (x < vtotal) {
                    int k = 0;
                    while (k + 1 < nseg && seg(k + 1)[plan::S_CHECK_OFF] <= x)
                        ++k;
                    const int *gg = seg(k);
                    const int nb = (k + 1 < nseg ? seg(k + 1)[plan::S_ID_OFF] : it[plan::I_IDS]) -
                                   gg[plan::S_ID_OFF];
                    const int local = x - gg[plan::S_CHECK_OFF];
                    const int m = local / nb, i = local % nb;
                    const bool shared = gg[plan::S_ROW_LO] == 0 && gg[plan::S_ROW_HI] == nrows && nmem > 1;
                    const int sq = shared ? members[m] : gg[plan::S_TABLE_SEQ];
                    got[u] = p.block_tables[(int64_t)sq * p.max_blocks_per_seq + gg[plan::S_BEGIN] / BS + i];
                    want[u] = ids[gg[plan::S_ID_OFF] + i];
                    kk4[u] = k;
                }
            }
        };
        auto fold_checks = [&]() {
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (kk4[u] >= 0 && got[u] != want[u])
                    segbad[kk4[u]] = 1;
        };
        // q rows as the B operand of S^T: [chunk][RQ rows][128 B], swizzled,
        // rows >= nrows zero
        constexpr int QPCS = D * 2 / 16;
        constexpr int QPER = (RQ * QPCS + NW * 32 - 1) / (NW * 32);
        uint4 qv[QPER];
        load_checks(0);
#pragma unroll
        for (int u = 0; u < QPER; ++u) {
            const int i = tid + u * NW * 32, r = i / QPCS;
            qv[u] = make_uint4(0u, 0u, 0u, 0u);
            if (i < RQ * QPCS && r < nrows && !invalid_item)
                qv[u] = reinterpret_cast<const uint4 *>(static_cast<const T *>(p.q) +
                                                        row_head(p, w, G, r) * D)[i % QPCS];
        }
        int m_exp = 0, m_plen = 0, m_len = 0;
        if (tid < nmem) {
            const int sq = members[tid];
            m_exp = expected[sq];
            m_plen = plan_lens[sq];
            m_len = p.context_lens[sq];
        }
        fold_checks();
#pragma unroll
        for (int u = 0; u < QPER; ++u) {
            const int i = tid + u * NW * 32;
            if (i < RQ * QPCS) {
                const int r = i / QPCS, pc = i % QPCS, c = pc / 8, q8 = pc % 8;
                *reinterpret_cast<uint4 *>(smem + CC::OFF_Q + c * CC::QPLANE + r * 128 +
                                           ((q8 ^ (r & 7)) << 4)) = qv[u];
            }
        }
        if (tid < nmem) {
            exp_s[tid] = m_exp;
            if (m_plen != m_len)
                atomicOr(lenbad, 1u << tid);
        }
        if (tid < RQ)
            mref[tid] = -INFINITY;
        for (int x0 = 4 * NW * 32; x0 < vtotal; x0 += 4 * NW * 32) {
            load_checks(x0);
            fold_checks();
        }
        fence_proxy_async_smem();   // q rows (generic stores) before the MMAs read them
        tc05::fence_before_sync();
        __syncthreads();

        // ---- the stages.  Warps 0 and 1 run the softmax of a stage's two
        // tiles (one token per lane); lane 0 of warp 2 issues the MMAs -- the
        // next stage's S^T as soon as this stage's scores are in registers,
        // this stage's O^T once its P is in shared memory; lane 0 of warp 3
        // refills the ring.
        float ls[CC::RPL];   // this lane's token's share of its rows' sums
#pragma unroll
        for (int j = 0; j < CC::RPL; ++j)
            ls[j] = 0.f;
        // M = 128 products take N a multiple of 16: the query rows' n-tiles
        // rounded up to 16 or 32 columns (the extra ones are never read)
        const int n16 = 16 * ((ntl + 1) / 2);
        const uint32_t id_qk = tc05::idesc<T>(128, n16, false, false);
        const uint32_t id_pv = tc05::idesc<T>(128, n16, true, true);
        const uint64_t q_desc = tc05::sdesc(qb, 16, 1024);
        // S^T of stage s into TMEM (the stage's K, A K-major; q rows, B K-major).
        // A is 128 rows of 8-row atoms 1 KiB apart from a chunk's first atom:
        // atom 4w is group w's K, so group w's 8 tokens land in TMEM lanes
        // 32w .. 32w + 7, warp w's quarter; the other rows are ignored.
        auto issue_qk = [&](int st) {
            const int gs = g + st, sl = gs % NSLOT;
            const uint64_t k_desc = tc05::sdesc(smem_u32(smem + CC::OFF_RING + sl * CC::SLOT), 16, 1024);
            if (!mbar_wait_bounded(&full[sl], (uint32_t)((gs / NSLOT) & 1))) {
                atomicOr(cta_flag, 2u);
                return;
            }
            tc05::fence_after_sync();
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint32_t off = (uint32_t)((ks / 4) * CC::ATOM + (ks % 4) * 32);
                const uint32_t qoff = (uint32_t)((ks / 4) * CC::QPLANE + (ks % 4) * 32);
                tc05::mma(tS, k_desc + (off >> 4), q_desc + (qoff >> 4), id_qk, ks > 0);
            }
            tc05::commit(sbar);
        };
        if (tid == kIssuer && n_st > 0)
            issue_qk(0);
        int k_use = 0;
        bool failed = false;
        int s = 0;
        for (; s < n_st; ++s) {
            const int gs = g + s, sl = gs % NSLOT;
            uint8_t *slot_p = smem + CC::OFF_RING + sl * CC::SLOT;
            bool bad = !mbar_wait_bounded(sbar, (uint32_t)(gs & 1));
            if (__syncthreads_or(bad || (*reinterpret_cast<volatile uint32_t *>(cta_flag) & 2u))) {
                failed = true;
                break;
            }
            tc05::fence_after_sync();

            // scores of this warp's group: tokens 8w .. 8w + 7 of the stage
            // (tile w / 2), read from lanes 0-7 of the warp's TMEM quarter and
            // shuffled out: lane = 8 rq + t takes token t's query rows
            // [RPL rq, RPL rq + RPL)
            const int tt = 2 * s + (warp >> 1), t = lane & 7, rq = lane >> 3;
            const int g_tok0 = (warp & 1) * CC::GRP;   // the group's first token in its tile
            int nvalid = 0, rlo = 0, rhi = 0;
            const bool tile_here = tt < total;
            if (tile_here) {
                const int k = seg_of(tt, k_use);
                const int *gg = seg(k);
                const int t0 = gg[plan::S_BEGIN] + (tt - gg[plan::S_FIRST_TILE]) * TILE;
                nvalid = min(TILE, gg[plan::S_END] - t0);
                rlo = gg[plan::S_ROW_LO];
                rhi = min(gg[plan::S_ROW_HI], nrows);
            }
            const bool valid = tile_here && g_tok0 + t < nvalid;
            float x[CC::RPL];
            {
                uint32_t sv[NT][8];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        sv[nt][j] = 0u;
                    if (nt < ntl)
                        tc05::ld8(tS + tlane + 8 * nt, sv[nt]);
                }
                tc05::wait_ld();
                float got[CC::RPL];
#pragma unroll
                for (int k = 0; k < 4; ++k)
#pragma unroll
                    for (int j = 0; j < CC::RPL; ++j) {
                        const int r = CC::RPL * k + j;
                        const uint32_t v = __shfl_sync(0xffffffffu, sv[r / 8][r % 8], t);
                        if (rq == k)
                            got[j] = __uint_as_float(v);
                    }
#pragma unroll
                for (int j = 0; j < CC::RPL; ++j) {
                    const int r = CC::RPL * rq + j;
                    const bool live = valid && r >= rlo && r < rhi;
                    x[j] = live ? got[j] * p.qscale : -INFINITY;
                }
            }
            bool over = false;
#pragma unroll
            for (int j = 0; j < CC::RPL; ++j)
                over |= x[j] > mref[CC::RPL * rq + j] + kSlack;
            tc05::fence_before_sync();
            const bool any_over = __syncthreads_or(over);
            // the scores are in registers: S^T may take the next stage
            if (tid == kIssuer && s + 1 < n_st)
                issue_qk(s + 1);
            // refill: stage s + NSLOT - 1 goes to the slot stage s - 1 used
            if (tid == kProducer && s + NSLOT - 1 < n_st) {
                bool ok = true;
                if (s >= 1) {
                    const int gp = gs - 1;
                    ok = mbar_wait_bounded(&empty[gp % NSLOT], (uint32_t)((gp / NSLOT) & 1));
                }
                if (ok) {
                    issue(s + NSLOT - 1);
                    *n_issued = s + NSLOT;
                } else {
                    atomicOr(cta_flag, 2u);
                }
            }
            if (any_over) {
                // exact running maxima: per warp over its 8 tokens (the lanes
                // of one rq), then over the warps in shared memory
#pragma unroll
                for (int j = 0; j < CC::RPL; ++j) {
                    float m8 = x[j];
                    m8 = fmaxf(m8, __shfl_xor_sync(0xffffffffu, m8, 1));
                    m8 = fmaxf(m8, __shfl_xor_sync(0xffffffffu, m8, 2));
                    m8 = fmaxf(m8, __shfl_xor_sync(0xffffffffu, m8, 4));
                    if (t == 0)
                        red[warp * RQ + CC::RPL * rq + j] = m8;
                }
                __syncthreads();
                auto stage_max = [&](int r) {
                    float mx = red[r];
#pragma unroll
                    for (int w2 = 1; w2 < NW; ++w2)
                        mx = fmaxf(mx, red[w2 * RQ + r]);
                    return mx;
                };
                bool grew = false;
#pragma unroll
                for (int j = 0; j < CC::RPL; ++j) {
                    const int r = CC::RPL * rq + j;
                    const float mo = mref[r], mn = fmaxf(mo, stage_max(r));
                    ls[j] *= mn == -INFINITY ? 1.f : exp2f(mo - mn);
                }
                for (int r = 0; r < RQ; ++r)
                    grew |= fmaxf(mref[r], stage_max(r)) != mref[r];
                __syncthreads();   // every thread has read the old references
                if (tid < RQ) {
                    const float mo = mref[tid], mn = fmaxf(mo, stage_max(tid));
                    alph[tid] = mn == -INFINITY ? 1.f : exp2f(mo - mn);
                    mref[tid] = mn;
                }
                __syncthreads();
                if (grew && s > 0) {
                    // O holds earlier stages: rescale it once their products
                    // are done (each warp its quarter of the dims)
                    const int gp = gs - 1;
                    bad = !mbar_wait_bounded(&empty[gp % NSLOT], (uint32_t)((gp / NSLOT) & 1));
                    if (!bad) {
                        tc05::fence_after_sync();
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            if (nt < ntl) {
                                uint32_t ov[8];
                                tc05::ld8(tO + tlane + 8 * nt, ov);
                                tc05::wait_ld();
#pragma unroll
                                for (int j = 0; j < 8; ++j)
                                    ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alph[8 * nt + j]);
                                tc05::st8(tO + tlane + 8 * nt, ov);
                            }
                        tc05::wait_st();
                    }
                }
                tc05::fence_before_sync();
                if (__syncthreads_or(bad)) {
                    failed = true;
                    ++s;   // the next stage's S^T may be in flight: drained below
                    break;
                }
            }
            // probabilities against the reference; P^T = hi + lo over the
            // group's K atoms as [token][query rows] (the B operand MN-major,
            // swizzled like the ring): this lane's RPL rows are RPL / 2
            // 32-bit words of token t's row
            {
                uint8_t *grp = slot_p + warp * CC::PERIOD;
#pragma unroll
                for (int i = 0; i < CC::RPL / 2; ++i) {
                    const int r = CC::RPL * rq + 2 * i;
                    const float a0 = x[2 * i] == -INFINITY ? 0.f : exp2f(x[2 * i] - fmaxf(mref[r], -1e30f));
                    const float a1 =
                        x[2 * i + 1] == -INFINITY ? 0.f : exp2f(x[2 * i + 1] - fmaxf(mref[r + 1], -1e30f));
                    ls[2 * i] += a0;
                    ls[2 * i + 1] += a1;
                    const uint32_t h = Mma<T>::pack(a0, a1);
                    const float2 hf = Mma<T>::unpack(h);
                    const uint32_t l = Mma<T>::pack(a0 - hf.x, a1 - hf.y);
                    const int byte = r * 2;
                    const int off = t * 128 + ((((byte >> 4) ^ t)) << 4) + (byte & 15);
                    *reinterpret_cast<uint32_t *>(grp + off) = h;
                    *reinterpret_cast<uint32_t *>(grp + CC::ATOM + off) = l;
                }
                // rows of V past the tile's valid tokens may hold anything (even
                // NaN patterns): zero them so that 0 * v stays 0
                if (tile_here && !valid && rq < CC::CHUNKS) {
                    uint4 *vrow = reinterpret_cast<uint4 *>(grp + CC::V_OFF + rq * CC::ATOM + t * 128);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        vrow[q] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            fence_proxy_async_smem();
            tc05::fence_before_sync();
            __syncthreads();
            if (tid == kIssuer) {
                tc05::fence_after_sync();
                const uint32_t sb = smem_u32(slot_p);
                const int nk = 2 * s + 1 < total ? 2 : 1;
                for (int j = 0; j < nk; ++j) {
                    // tokens 16j .. 16j + 15: groups 2j, 2j + 1, one period apart;
                    // V^T MN-major (chunks one atom apart), P^T MN-major
                    const uint32_t gb = sb + (uint32_t)(2 * j * CC::PERIOD);
                    const uint64_t a = tc05::sdesc(gb + CC::V_OFF, CC::ATOM, CC::PERIOD);
                    tc05::mma(tO, a, tc05::sdesc(gb, CC::PERIOD, CC::PERIOD), id_pv, s > 0 || j > 0);
                    tc05::mma(tO, a, tc05::sdesc(gb + CC::ATOM, CC::PERIOD, CC::PERIOD), id_pv, true);
                }
                tc05::commit(&empty[sl]);
            }
        }
        const int done_st = s;   // stages whose S^T was consumed (failed: maybe fewer)
        if (failed) {
            // let the copies and products in flight finish before the memory
            // they write is reused or released
            if (tid == 0) {
                report(p.status, PKV_DEV_TIMEOUT);
                atomicOr(cta_flag, 1u);
            }
            const int issued = *reinterpret_cast<volatile int32_t *>(n_issued);
            for (int i = done_st; i < issued && i < n_st; ++i) {
                const int gi = g + i;
                drain_wait(&full[gi % NSLOT], (uint32_t)((gi / NSLOT) & 1), p.status);
            }
            if (done_st < n_st)   // an S^T issued for a stage not consumed
                drain_wait(sbar, (uint32_t)((g + done_st) & 1), p.status);
            if (done_st > 0)
                drain_wait(&empty[(g + done_st - 1) % NSLOT],
                           (uint32_t)(((g + done_st - 1) / NSLOT) & 1), p.status);
        } else if (n_st > 0) {
            // every product of the item done (one commit covers all before it)
            const int gl = g + n_st - 1;
            if (!mbar_wait_bounded(&empty[gl % NSLOT], (uint32_t)((gl / NSLOT) & 1))) {
                if (tid == 0) {
                    report(p.status, PKV_DEV_TIMEOUT);
                    atomicOr(cta_flag, 1u);
                }
            }
            tc05::fence_after_sync();
        }
        g += n_st;

        // ---- row sums over the tokens' lanes, bad rows, results
        // row sums: over a warp's 8 token lanes, then over the warps
#pragma unroll
        for (int j = 0; j < CC::RPL; ++j) {
            float sm = ls[j];
            sm += __shfl_xor_sync(0xffffffffu, sm, 1);
            sm += __shfl_xor_sync(0xffffffffu, sm, 2);
            sm += __shfl_xor_sync(0xffffffffu, sm, 4);
            if ((lane & 7) == 0)
                red[warp * RQ + CC::RPL * (lane >> 3) + j] = sm;
        }
        if (tid == 0) {
            bool any = invalid_item;
            uint32_t mask = 0;
            for (int k = 0; k < nseg && k < CC::MAXSEG; ++k)
                if (segbad[k]) {
                    any = true;
                    for (int r = seg(k)[plan::S_ROW_LO]; r < seg(k)[plan::S_ROW_HI] && r < 32; ++r)
                        mask |= 1u << r;
                }
            const uint32_t lb = *lenbad;
            for (int mm = 0; mm < nmem; ++mm)
                if ((lb >> mm) & 1u)
                    mask |= ((1u << G) - 1u) << (mm * G);
            *badrows = mask;
            if (any)
                report(p.status, PKV_DEV_BAD_BLOCK);
            if (lb)
                report(p.status, PKV_DEV_BAD_CONTEXT_LEN);
        }
        __syncthreads();
        const bool failed_all = invalid_item || failed || n_st == 0 ||
                                *reinterpret_cast<volatile uint32_t *>(cta_flag) != 0;
        // O^T: this thread's dim d = 32 warp + lane, one register per row
        float o[RQ];
#pragma unroll
        for (int r = 0; r < RQ; ++r)
            o[r] = 0.f;
        if (!failed_all) {
            uint32_t ov[NT][8];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                if (nt < ntl)
                    tc05::ld8(tO + tlane + 8 * nt, ov[nt]);
            tc05::wait_ld();
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (nt < ntl)
                        o[8 * nt + j] = __uint_as_float(ov[nt][j]);
        }
        const int d = 32 * warp + lane;
#pragma unroll
        for (int r = 0; r < RQ; ++r) {
            if (r < nrows) {
                const bool bad_r = failed_all || ((*badrows >> r) & 1u);
                const float L = red[r] + red[RQ + r] + red[2 * RQ + r] + red[3 * RQ + r];
                const int64_t sh = row_head(p, w, G, r);
                if (exp_s[r / G] == 1) {
                    const float inv = !bad_r && L > 0.f ? 1.f / L : 0.f;
                    store_out(p.out, p.out_dtype, sh * D + d, bad_r ? 0.f : o[r] * inv);
                } else {
                    __stcg(p.ws_acc + (sh * slots + slot) * D + d, bad_r ? 0.f : o[r]);
                    if (d == 0)
                        __stcg(reinterpret_cast<float2 *>(p.ws_ml) + sh * slots + slot,
                               make_float2(bad_r ? -INFINITY : mref[r], bad_r ? -1.f : L));
                }
            }
        }
        tc05::fence_before_sync();
        __syncthreads();
        tc05::fence_after_sync();
        item = next;
    }
    tc05::fence_before_sync();
    __syncthreads();
    if (warp == 0)
        tc05::dealloc(*tslot, CC::TM_COLS);
}

}  // namespace pkv
