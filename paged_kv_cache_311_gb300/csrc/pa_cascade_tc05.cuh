// pa_cascade_tc05.cuh -- shared-prefix (cascade) decode on the 5th-generation
// tensor cores (tcgen05), one warp-specialised CTA per SM.
//
// Same plan, items, device checks, outputs and partials as pa_cascade_kernel
// (cascade_plan.h; PagedAttention: Efficient LLM Serving with vLLM,
// "Advanced Features", KV-Cache Sharing): for every row of an item (query
// head h of member m), the softmax-weighted sum of V over the item's tokens,
// written as the output when the item holds the sequence entirely, else as
// an unnormalised partial (max, sum, acc) for pa_cascade_merge_kernel.
//
// Work: the plan's (list, kv head) units are dealt round-robin to one CTA
// per SM; a CTA walks its units' items one after the other.  Each item's
// 16-token tiles are grouped into stages of 128 tokens (8 tiles; an item's
// last stage may be partly empty).  Roles, one CTA:
//   * loader warp: copies the next item's record into a two-slot record
//     ring, then stages its query rows (the B operand of S^T), then runs the
//     device checks (block ids in range and equal to the device tables,
//     lengths equal to the plan's), each step released on its own barrier;
//   * producer warp: TMA loads of each stage's K and V (one box per block
//     piece and 64-element chunk plane, the 32 lanes issuing in parallel)
//     into a three-stage ring;
//   * MMA thread: S^T = K q^T (M = 128 tokens, N = 32 query-row columns,
//     K = 128 dims) into one of two TMEM score buffers, then O^T += V^T P^T
//     for the stage before (M = 128 dims, N = 32, K = the stage's valid
//     16-token tiles) into one TMEM accumulator; each completion is
//     signalled with tcgen05.commit on a per-stage mbarrier;
//   * twelve softmax warps, four per group of 8 query rows (one per TMEM
//     lane quarter): thread = one token of the stage, for its group's rows.  Online softmax in the log2 domain against a reference maximum
//     per query row shared by the CTA, kept while every new score stays
//     within 2^8 of it (a per-stage OR over the four warps); otherwise the
//     exact stage maxima (warp shuffles, then shared memory) move the
//     references and O is rescaled in TMEM.  P = hi + lo 16-bit parts, so the
//     products keep fp32-level accuracy, written over the stage's K (used
//     by then) as [token][hi rows | lo rows], one N = 64 B operand read
//     MN-major (high and low products land in separate O^T columns).  At the
//     end of an item the same warps read O^T (thread = one dim) and write
//     the rows' outputs or partials.
// Every hand-off is an mbarrier phase (K, V full; scores full / free; P full;
// stage free; record, q rows, checks full; record free), so no role waits for another's slowest
// warp, and the next item's loads stream while an item's epilogue runs.
// Every wait is bounded (PKV_DEV_TIMEOUT); the softmax warps take their
// decisions together through a named-barrier OR.
#pragma once

#include "pa_cascade.cuh"

namespace pkv {

template <typename T, int D, int BS, int G>
struct Tc05Cfg {
    static_assert(D == 128, "the tcgen05 cascade kernel takes head_dim 128");
    static constexpr int TILE = plan::kTileTokens;   // 16 tokens
    static constexpr int TOK = 128;                  // tokens per stage: M of S^T
    static constexpr int TPS = TOK / TILE;           // tiles per stage
    static constexpr int NSTAGE = 3;
    static constexpr int PLANE = TOK * 128;          // one 64-element chunk of a stage's rows
    static constexpr int KV_BYTES = 2 * PLANE;       // K (or V) of one stage
    static constexpr int STAGE = 2 * KV_BYTES;       // K then V
    static constexpr int RQ = plan::kMaxRows;        // query rows of an item (24)
    static constexpr int N = 32;                     // MMA N: the rows padded to 32
    static constexpr int QPLANE = N * 128;
    static constexpr int QBUF = 2 * QPLANE;          // q rows of one item: [chunk][32 rows][128 B]
    static constexpr int BOX_ROWS = BS < TILE ? BS : TILE;
    static constexpr int BOX_BYTES = BOX_ROWS * 128; // one box: BOX_ROWS rows of one chunk
    static constexpr int MAXSEG = plan::max_segments(G);
    static constexpr int ITEM_INTS = plan::item_ints(G);
    static constexpr int IDS = plan::item_ids_offset(G);
    static constexpr int SEGS = plan::item_segments_offset();
    static constexpr int TABLE_CAP = plan::kTableCap;
    // an item's slot of the record ring: what the loader worked out (the M_*
    // ints), the record, then per-segment bad flags and the members' expected
    // partial counts
    enum { M_NST = 0, M_END, M_FAILED, M_ZERO, M_BADROWS, M_KVH, M_FINAL, M_HEAD };
    static constexpr int META_INTS = M_HEAD + ITEM_INTS + MAXSEG + RQ;
    static constexpr int META_BYTES = (META_INTS * 4 + 15) / 16 * 16;
    static constexpr int OFF_Q = NSTAGE * STAGE;
    static constexpr int OFF_META = OFF_Q + 2 * QBUF;
    static constexpr int OFF_RED = OFF_META + 2 * META_BYTES;   // [2][4 warps][32 rows] floats
    static constexpr int OFF_BAR = OFF_RED + 2 * 4 * N * 4;
    enum {
        B_KFULL = 0,
        B_VFULL = B_KFULL + NSTAGE,
        B_SFULL = B_VFULL + NSTAGE,
        B_SFREE = B_SFULL + 2,
        B_PFULL = B_SFREE + 2,
        B_STFREE = B_PFULL + NSTAGE,
        B_RECFULL = B_STFREE + NSTAGE,
        B_QFULL = B_RECFULL + 2,
        B_METAFULL = B_QFULL + 2,
        B_RECEMPTY = B_METAFULL + 2,
        B_MMADONE = B_RECEMPTY + 2,
        B_DONE = B_MMADONE + 1,
        NBAR = B_DONE + 1
    };
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;   // TMEM address, abort flag
    static constexpr int SMEM_USED = OFF_MISC + 16;
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;   // slack for 1024-byte alignment
    // softmax warps: three row groups (query rows 8j .. 8j + 7) of four warps,
    // one per TMEM lane quarter
    static constexpr int NRG = RQ / 8;
    static constexpr int SWARPS = 4 * NRG;
    static constexpr int WARPS = 3 + SWARPS;              // producer, MMA, loader, softmax
    static constexpr int THREADS = WARPS * 32;
    // TMEM columns: S^T buffer b in two partial sums (even / odd 16-dim
    // k-steps) at 64 b and 64 b + 32; O^T in two partial sums (even / odd
    // 16-token tile) of 64 columns at 128 + 64 k, each [P's high part rows
    // 0-31 | low part rows 0-31]
    static constexpr int TM_COLS = 256;
    static constexpr int TM_O = 128;
    static constexpr int kRecEmptyArrivals = 2 + SWARPS;  // producer, MMA commit, softmax warps
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static_assert(PLANE % 1024 == 0 && STAGE % 1024 == 0 && OFF_Q % 1024 == 0 && QPLANE % 1024 == 0,
                  "128-byte swizzle atoms are 1024-byte aligned");
    static_assert(BOX_ROWS % 8 == 0, "boxes start on 8-row atoms");
    static_assert(RQ <= N && RQ % 8 == 0 && RQ <= 32, "query rows");
};

// Named barrier of the twelve softmax warps (id 1, 384 threads): a sync, and
// an OR of one predicate over them.
__device__ __forceinline__ void softmax_sync()
{
    __syncwarp();
    asm volatile("bar.sync 1, 384;" ::: "memory");
}
__device__ __forceinline__ bool softmax_any(bool v)
{
    uint32_t r;
    __syncwarp();
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
                 "bar.red.or.pred p, 1, 384, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(r)
                 : "r"((uint32_t)v)
                 : "memory");
    return r != 0;
}

// 2^x, the special-function unit's approximation (relative error far below
// the 2^-16 of the P split it feeds)
__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <typename T, int D, int BS, int G>
__global__ void __launch_bounds__(Tc05Cfg<T, D, BS, G>::THREADS, 1)
pa_cascade_tc05_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv, const int32_t *plan_buf, int num_lists)
{
    using CC = Tc05Cfg<T, D, BS, G>;
    constexpr int NSTAGE = CC::NSTAGE, RQ = CC::RQ, TILE = CC::TILE, TPS = CC::TPS;
    constexpr float kSlack = 8.f;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = aligned_smem(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + CC::OFF_BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + CC::OFF_MISC);
    uint32_t *abort_flag = tslot + 1;

    const int B = p.num_seqs, slots = p.num_partitions, Hk = p.num_kv_heads;
    const int32_t *expected = plan_buf + plan::kHeader;
    const int32_t *plan_lens = expected + B;
    const int32_t *items = plan_buf + plan::kHeader + 2 * B;

    if (tid == 0) {
        for (int i = 0; i < NSTAGE; ++i) {
            mbar_init(&bars[CC::B_KFULL + i], 1);
            mbar_init(&bars[CC::B_VFULL + i], 1);
            mbar_init(&bars[CC::B_PFULL + i], CC::SWARPS);
            mbar_init(&bars[CC::B_STFREE + i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[CC::B_SFULL + i], 1);
            mbar_init(&bars[CC::B_SFREE + i], CC::SWARPS);
            mbar_init(&bars[CC::B_RECFULL + i], 1);
            mbar_init(&bars[CC::B_QFULL + i], 1);
            mbar_init(&bars[CC::B_METAFULL + i], 1);
            mbar_init(&bars[CC::B_RECEMPTY + i], CC::kRecEmptyArrivals);
        }
        mbar_init(&bars[CC::B_MMADONE], 1);
        mbar_init(&bars[CC::B_DONE], CC::WARPS);
        fence_mbar_init();
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
        *abort_flag = 0;
    }
    if (warp == 1)
        tc05::alloc(tslot, CC::TM_COLS);
    tc05::fence_before_sync();
    __syncthreads();
    tc05::fence_after_sync();
    const uint32_t tS = *tslot, tO = tS + CC::TM_O;
    // launched as a programmatic dependent of the previous kernel: nothing it
    // may write is read before this wait; then the merge kernel behind this
    // grid may start (it reads the plan before its own wait)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    auto meta = [&](int b) { return reinterpret_cast<int32_t *>(smem + CC::OFF_META + b * CC::META_BYTES); };
    auto rec_of = [&](int32_t *m) { return m + CC::M_HEAD; };
    auto segbad_of = [&](int32_t *m) { return m + CC::M_HEAD + CC::ITEM_INTS; };
    auto exp_of = [&](int32_t *m) { return m + CC::M_HEAD + CC::ITEM_INTS + CC::MAXSEG; };
    auto aborted = [&]() { return *reinterpret_cast<volatile uint32_t *>(abort_flag) != 0; };
    // a bounded wait; giving up stops the CTA's work (every role sees the flag)
    auto wait = [&](int bar, uint32_t parity) {
        if (mbar_wait_bounded(&bars[bar], parity))
            return true;
        if (atomicOr(abort_flag, 1u) == 0)
            report(p.status, PKV_DEV_TIMEOUT);
        return false;
    };
    // the same, polling with the non-blocking test and a short back-off, for
    // the pipeline's hand-offs (a suspended try_wait resumed measurably late)
    auto wait_poll = [&](int bar, uint32_t parity) {
        if (mbar_test_wait(&bars[bar], parity))
            return true;
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t it = 1;; ++it) {
            __nanosleep(20);
            if (mbar_test_wait(&bars[bar], parity))
                return true;
            if ((it & 63u) == 0 && (globaltimer_ns() - t0 > kWaitLimitNs || it >= (1u << 30))) {
                if (atomicOr(abort_flag, 1u) == 0)
                    report(p.status, PKV_DEV_TIMEOUT);
                return false;
            }
        }
    };

    if (warp == 0) {
        // ------------------------------------------------------- producer
        // The warp issues a stage's loads together: lane 4u + 2c + v takes
        // tile u of the stage, 64-dim chunk plane c, K (v = 0) or V (v = 1),
        // and issues that plane's box(es) of the tile (one thread issuing
        // every box of a stage was measured at ~120 ns per box, the
        // pipeline's limit).
        const int u = lane >> 2, c = (lane >> 1) & 1, v = lane & 1;
        const CUtensorMap *map = v ? &tmv : &tmk;
        int g = 0;
        for (int n = 0;; ++n) {
            const int b = n & 1;
            const bool okr = wait(CC::B_RECFULL + b, (uint32_t)((n >> 1) & 1));
            if (!__all_sync(0xffffffffu, okr))
                break;
            int32_t *m = meta(b);
            if (m[CC::M_END])
                break;
            const int32_t *it = rec_of(m);
            const int n_st = m[CC::M_NST], kvh = m[CC::M_KVH];
            const int nseg = it[plan::I_NSEG], total = it[plan::I_TILES];
            const int32_t *ids = it + CC::IDS;
            auto seg = [&](int k) { return it + CC::SEGS + plan::kSegInts * k; };
            int kcur = 0;
            bool stop = false;
            for (int s = 0; s < n_st; ++s, ++g) {
                const int slot = g % NSTAGE;
                const bool oks = g < NSTAGE || wait_poll(CC::B_STFREE + slot, (uint32_t)(((g / NSTAGE) - 1) & 1));
                if (!__all_sync(0xffffffffu, oks)) {
                    stop = true;
                    break;
                }
                // this lane's tile: its token range and boxes
                const int tile = TPS * s + u;
                int t0 = 0, te = 0, sid = 0, sb0 = 0;
                if (tile < total) {
                    while (kcur + 1 < nseg && seg(kcur + 1)[plan::S_FIRST_TILE] <= tile)
                        ++kcur;
                    const int *gg = seg(kcur);
                    t0 = gg[plan::S_BEGIN] + (tile - gg[plan::S_FIRST_TILE]) * TILE;
                    te = min(gg[plan::S_END], t0 + TILE);
                    sid = gg[plan::S_ID_OFF];
                    sb0 = gg[plan::S_BEGIN] / BS;
                }
                const int nbox = (te - t0 + CC::BOX_ROWS - 1) / CC::BOX_ROWS;
                // bytes each of K and V: the boxes of every tile, both planes
                const uint32_t bytes = __reduce_add_sync(0xffffffffu, (c == 0 && v == 0) ? (uint32_t)nbox : 0u) *
                                       (uint32_t)(2 * CC::BOX_BYTES);
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bars[CC::B_KFULL + slot], bytes);
                    mbar_arrive_expect_tx(&bars[CC::B_VFULL + slot], bytes);
                }
                __syncwarp();
                uint8_t *dst = smem + slot * CC::STAGE + v * CC::KV_BYTES + c * CC::PLANE + u * TILE * 128;
                uint64_t *bar = &bars[(v ? CC::B_VFULL : CC::B_KFULL) + slot];
                for (int bx = 0; bx < nbox; ++bx) {
                    const int tok = t0 + bx * CC::BOX_ROWS;
                    int phys = ids[sid + tok / BS - sb0];
                    if (phys < 0 || (int64_t)phys >= p.num_blocks)
                        phys = 0;   // flagged by the loader's checks
                    tma_load_5d(dst + bx * CC::BOX_BYTES, map, bar, 0, tok % BS, c, kvh, phys);
                }
            }
            if (stop)
                break;
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars[CC::B_RECEMPTY + b]);
        }
        // no load may still be writing the ring when the CTA leaves: the
        // last stage issued into each slot has landed (in normal runs the
        // consumers already waited for every one of them)
        if (lane == 0) {
            for (int x = g - NSTAGE < 0 ? 0 : g - NSTAGE; x < g; ++x) {
                drain_wait(&bars[CC::B_KFULL + x % NSTAGE], (uint32_t)((x / NSTAGE) & 1), p.status);
                drain_wait(&bars[CC::B_VFULL + x % NSTAGE], (uint32_t)((x / NSTAGE) & 1), p.status);
            }
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA
        // One thread, an event loop: the PV of the oldest stage whose P is
        // written (it frees that ring slot for the producer), else the S^T of
        // the next stage once its K has landed and its score buffer is free.
        // Neither waits for the other, so a slot is held only from its load
        // to its PV.
        if (lane == 0) {
            const uint32_t id_qk = tc05::idesc<T>(128, CC::N, false, false);
            // O^T gets P's high and low parts in one product: N = 64 columns,
            // the low part's rows 32 columns after the high part's
            const uint32_t id_pv = tc05::idesc<T>(128, 2 * CC::N, true, true);
            int gq = 0, gp = 0;                  // stages with S^T issued / with PV issued
            int pk[4] = {0, 0, 0, 0};            // per issued stage (gq - gp <= 2): valid tiles,
            bool pf[4] = {false, false, false, false};   // and whether it starts its item
            int n = 0, cur_b = 0, q_s = 0, q_nst = -1, q_total = 0;
            uint32_t qb = 0;
            bool items_done = false, ok = true;
            uint64_t t_idle = 0;
            for (uint32_t spin = 0;; ++spin) {
                bool progress = false;
                if (gp < gq) {
                    const int slot = gp % NSTAGE;
                    const uint32_t par = (uint32_t)((gp / NSTAGE) & 1);
                    if (mbar_test_wait(&bars[CC::B_PFULL + slot], par) &&
                        mbar_test_wait(&bars[CC::B_VFULL + slot], par)) {
                        // O^T += V^T P^T over the stage's valid tiles: A = V^T
                        // MN-major (64-dim chunk planes PLANE apart, 8-token
                        // groups 1 KiB apart), B = P^T MN-major over the stage's
                        // K, a token's 128-byte row [hi rows 0-31 | lo rows 0-31]
                        tc05::fence_after_sync();
                        const uint32_t kb = smem_u32(smem + slot * CC::STAGE), vb = kb + CC::KV_BYTES;
                        const int nk = pk[gp & 3];
                        for (int k = 0; k < nk; ++k) {
                            // the item's first stage starts each partial sum
                            const bool acc = !(pf[gp & 3] && k < 2);
                            const uint64_t a = tc05::sdesc(vb + k * 2048, CC::PLANE, 1024);
                            const uint64_t bp = tc05::sdesc(kb + k * 2048, CC::PLANE, 1024);
                            tc05::mma(tO + 64 * (k & 1), a, bp, id_pv, acc);
                        }
                        tc05::commit(&bars[CC::B_STFREE + slot]);
                        ++gp;
                        progress = true;
                    }
                }
                if (!items_done && q_nst < 0) {
                    // the next item's q rows (every item releases its record
                    // slot once its S^T products have read them)
                    const int b = n & 1;
                    if (mbar_test_wait(&bars[CC::B_QFULL + b], (uint32_t)((n >> 1) & 1))) {
                        int32_t *m = meta(b);
                        ++n;
                        progress = true;
                        if (m[CC::M_END]) {
                            items_done = true;
                        } else if (m[CC::M_NST] == 0) {
                            tc05::commit(&bars[CC::B_RECEMPTY + b]);
                        } else {
                            cur_b = b;
                            q_nst = m[CC::M_NST];
                            q_total = rec_of(m)[plan::I_TILES];
                            q_s = 0;
                            qb = smem_u32(smem + CC::OFF_Q + b * CC::QBUF);
                        }
                    }
                }
                if (q_nst > 0 && gq - gp < 2) {
                    const int slot = gq % NSTAGE, sb = gq & 1;
                    if (mbar_test_wait(&bars[CC::B_KFULL + slot], (uint32_t)((gq / NSTAGE) & 1)) &&
                        (gq < 2 || mbar_test_wait(&bars[CC::B_SFREE + sb], (uint32_t)(((gq >> 1) - 1) & 1)))) {
                        // S^T = K q^T: both operands K-major, 128-byte swizzled;
                        // a 16-dim k-step moves 32 bytes along the row, the
                        // second 64-dim chunk is the next plane
                        tc05::fence_after_sync();
                        const uint32_t kb = smem_u32(smem + slot * CC::STAGE);
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks) {
                            const uint64_t a = tc05::sdesc(kb + (ks / 4) * CC::PLANE + (ks % 4) * 32, 16, 1024);
                            const uint64_t bq = tc05::sdesc(qb + (ks / 4) * CC::QPLANE + (ks % 4) * 32, 16, 1024);
                            tc05::mma(tS + sb * 64 + 32 * (ks & 1), a, bq, id_qk, ks > 1);
                        }
                        tc05::commit(&bars[CC::B_SFULL + sb]);
                        pk[gq & 3] = min(TPS, q_total - TPS * q_s);
                        pf[gq & 3] = q_s == 0;
                        ++gq;
                        progress = true;
                        if (++q_s == q_nst) {
                            tc05::commit(&bars[CC::B_RECEMPTY + cur_b]);   // its q rows are read
                            q_nst = -1;
                        }
                    }
                }
                if (items_done && gp == gq)
                    break;
                // bounded: give up after the wait limit without any progress;
                // idle polls back off briefly so that the softmax warp on this
                // SM sub-partition keeps its issue slots
                if (progress) {
                    t_idle = 0;
                    continue;
                }
                __nanosleep(32);
                if ((spin & 63u) == 0) {
                    const uint64_t now = globaltimer_ns();
                    if (t_idle == 0) {
                        t_idle = now;
                    } else if (now - t_idle > kWaitLimitNs || aborted()) {
                        if (atomicOr(abort_flag, 1u) == 0)
                            report(p.status, PKV_DEV_TIMEOUT);
                        ok = false;
                        break;
                    }
                }
            }
            (void)ok;
            // every product done before the TMEM goes
            tc05::commit(&bars[CC::B_MMADONE]);
            drain_wait(&bars[CC::B_MMADONE], 0u, p.status);
        }
    } else if (warp == 2) {
        // -------------------------------------------------------- loader
        // Per item, in order: the record (-> RECFULL: the producer and the
        // softmax warps may start), the query rows (-> QFULL: the MMA may
        // start), the device checks and the members' partial counts
        // (-> METAFULL: needed by the item's epilogue).
        const int units = Hk * num_lists;
        constexpr int RPL = (CC::ITEM_INTS + 31) / 32;   // record ints per lane
        int n = 0;
        bool stop = false;
        auto next_slot = [&]() {
            const int b = n & 1;
            if (n >= 2 && !wait(CC::B_RECEMPTY + b, (uint32_t)(((n >> 1) - 1) & 1)))
                return -1;
            return b;
        };
        for (int un = blockIdx.x; un < units && !stop; un += gridDim.x) {
            const int kvh = un % Hk;
            for (int item = un / Hk; item >= 0 && item < p.num_items;) {
                // the record's loads leave before the wait for its slot
                int32_t rv[RPL];
                const int32_t *src = items + (int64_t)item * CC::ITEM_INTS;
#pragma unroll
                for (int k = 0; k < RPL; ++k) {
                    const int i = lane + 32 * k;
                    rv[k] = i < CC::ITEM_INTS ? src[i] : 0;
                }
                const int b = next_slot();
                if (b < 0) {
                    stop = true;
                    break;
                }
                int32_t *m = meta(b);
                int32_t *it = rec_of(m);
                int32_t *segbad = segbad_of(m);
                int32_t *exps = exp_of(m);
#pragma unroll
                for (int k = 0; k < RPL; ++k) {
                    const int i = lane + 32 * k;
                    if (i < CC::ITEM_INTS)
                        it[i] = rv[k];
                }
                if (lane < CC::MAXSEG)
                    segbad[lane] = 0;
                __syncwarp();
                const int nseg = it[plan::I_NSEG], total = it[plan::I_TILES], nrows = it[plan::I_NROWS];
                const int nxt = it[plan::I_NEXT] > item && it[plan::I_NEXT] < p.num_items ? it[plan::I_NEXT] : -1;
                const bool invalid = nseg > 0 && (it[plan::I_IDS] > CC::TABLE_CAP || nseg > CC::MAXSEG ||
                                                  nrows > RQ || nrows <= 0 || total <= 0);
                const bool dead = aborted();
                const int n_st = (nseg <= 0 || invalid || dead) ? 0 : (total + TPS - 1) / TPS;
                if (lane == 0) {
                    m[CC::M_NST] = n_st;
                    m[CC::M_END] = 0;
                    m[CC::M_FAILED] = invalid || dead;
                    m[CC::M_ZERO] = nseg <= 0;
                    m[CC::M_BADROWS] = 0;
                    m[CC::M_FINAL] = nseg <= 0 ? -1 : 0;
                    m[CC::M_KVH] = kvh;
                    mbar_arrive(&bars[CC::B_RECFULL + b]);   // the producer and softmax may start
                }
                const int nmem = nrows > 0 && nrows <= RQ ? nrows / G : 0;
                const int32_t *members = it + plan::kItemHead;
                const CtaWork w{it[plan::I_SEQ0], nrows, kvh, 0, 0, it[plan::I_SLOT], it[plan::I_SEQ0], members};
                if (n_st > 0) {
                    // q rows -> [chunk][32 rows][128 B], 128-byte swizzled, and
                    // the members' expected partial counts and lengths: all
                    // loads in flight before the first store
                    uint8_t *qs = smem + CC::OFF_Q + b * CC::QBUF;
                    constexpr int PCS = D * 2 / 16;   // 16-byte pieces per row
                    constexpr int PER = (RQ * PCS + 31) / 32;
                    uint4 qv[PER];
#pragma unroll
                    for (int k = 0; k < PER; ++k) {
                        const int i = lane + 32 * k, r = i / PCS;
                        qv[k] = make_uint4(0u, 0u, 0u, 0u);
                        if (r < nrows)
                            qv[k] = reinterpret_cast<const uint4 *>(static_cast<const T *>(p.q) +
                                                                    row_head(p, w, G, r) * D)[i % PCS];
                    }
                    int m_exp = 0, m_plen = 0, m_len = 0;
                    if (lane < nmem) {
                        const int sq = members[lane];
                        m_exp = expected[sq];
                        m_plen = plan_lens[sq];
                        m_len = p.context_lens[sq];
                    }
#pragma unroll
                    for (int k = 0; k < PER; ++k) {
                        const int i = lane + 32 * k;
                        if (i < RQ * PCS) {
                            const int r = i / PCS, pc = i % PCS, ch = pc / 8, q8 = pc % 8;
                            *reinterpret_cast<uint4 *>(qs + ch * CC::QPLANE + r * 128 + ((q8 ^ (r & 7)) << 4)) = qv[k];
                        }
                    }
                    fence_proxy_async_smem();   // the q rows (generic stores) before the MMAs read them
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&bars[CC::B_QFULL + b]);
                    if (lane < nmem)
                        exps[lane] = m_exp;
                    const uint32_t lb = __reduce_or_sync(0xffffffffu, (lane < nmem && m_plen != m_len) ? 1u << lane : 0u);
                    // device checks, all loads of a round in flight together
                    const int vtotal = it[plan::I_CHECKS];
                    auto seg = [&](int k) { return it + CC::SEGS + plan::kSegInts * k; };
                    for (int x0 = 0; x0 < vtotal; x0 += 32 * 8) {
                        int got[8], want[8], kk[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const int x = x0 + 32 * k + lane;
                            kk[k] = -1;
                            got[k] = want[k] = 0;
                            if (x < vtotal) {
                                int sg = 0;
                                while (sg + 1 < nseg && seg(sg + 1)[plan::S_CHECK_OFF] <= x)
                                    ++sg;
                                const int *gg = seg(sg);
                                const int nb = (sg + 1 < nseg ? seg(sg + 1)[plan::S_ID_OFF] : it[plan::I_IDS]) -
                                               gg[plan::S_ID_OFF];
                                const int local = x - gg[plan::S_CHECK_OFF];
                                const int mi = local / nb, i = local % nb;
                                const bool shared = gg[plan::S_ROW_LO] == 0 && gg[plan::S_ROW_HI] == nrows &&
                                                    nmem > 1;
                                const int sq = shared ? members[mi] : gg[plan::S_TABLE_SEQ];
                                got[k] = p.block_tables[(int64_t)sq * p.max_blocks_per_seq +
                                                        gg[plan::S_BEGIN] / BS + i];
                                want[k] = it[CC::IDS + gg[plan::S_ID_OFF] + i];
                                kk[k] = sg;
                            }
                        }
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            if (kk[k] >= 0 && (got[k] != want[k] || want[k] < 0 ||
                                               (int64_t)want[k] >= p.num_blocks))
                                segbad[kk[k]] = 1;
                    }
                    __syncwarp();
                    if (lane == 0) {
                        bool any = false;
                        uint32_t mask = 0;
                        for (int k = 0; k < nseg; ++k)
                            if (segbad[k]) {
                                any = true;
                                for (int r = seg(k)[plan::S_ROW_LO]; r < seg(k)[plan::S_ROW_HI] && r < 32; ++r)
                                    mask |= 1u << r;
                            }
                        for (int mi = 0; mi < nmem; ++mi)
                            if ((lb >> mi) & 1u)
                                mask |= ((1u << G) - 1u) << (mi * G);
                        m[CC::M_BADROWS] = (int32_t)mask;
                        uint32_t fin = 0;   // rows whose sequence the item holds entirely
                        for (int r = 0; r < nrows; ++r)
                            if (exps[r / G] == 1)
                                fin |= 1u << r;
                        m[CC::M_FINAL] = (int32_t)fin;
                        if (any)
                            report(p.status, PKV_DEV_BAD_BLOCK);
                        if (lb)
                            report(p.status, PKV_DEV_BAD_CONTEXT_LEN);
                    }
                } else {
                    if (nseg <= 0) {
                        if (lane == 0 && kvh == 0) {
                            const int L = p.context_lens[it[plan::I_SEQ0]];
                            if (L < 0 || L > p.max_context_len)
                                report(p.status, PKV_DEV_BAD_CONTEXT_LEN);
                        }
                    } else {
                        // an item the CTA cannot run (a malformed record, or the
                        // CTA gave up after a timeout): its rows fail
                        if (lane < nmem)
                            exps[lane] = expected[members[lane]];
                        __syncwarp();
                        if (lane == 0) {
                            m[CC::M_BADROWS] = -1;
                            uint32_t fin = 0;
                            for (int r = 0; r < nrows && r < RQ; ++r)
                                if (exps[r / G] == 1)
                                    fin |= 1u << r;
                            m[CC::M_FINAL] = (int32_t)fin;
                            if (invalid)
                                report(p.status, PKV_DEV_BAD_BLOCK);
                        }
                    }
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&bars[CC::B_QFULL + b]);
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&bars[CC::B_METAFULL + b]);
                ++n;
                item = nxt;
            }
        }
        if (!stop) {
            const int b = next_slot();
            if (b >= 0 && lane == 0) {
                meta(b)[CC::M_END] = 1;
                mbar_arrive(&bars[CC::B_RECFULL + b]);
                mbar_arrive(&bars[CC::B_QFULL + b]);
                mbar_arrive(&bars[CC::B_METAFULL + b]);
            }
        }
    } else {
        // ------------------------------------------------------- softmax
        const int sw = warp - 3;                    // softmax warp 0 .. SWARPS - 1
        const int j = sw >> 2;                      // row group: query rows 8j .. 8j + 7
        const int r0 = 8 * j;
        const int qw = warp & 3;                    // TMEM lane quarter
        const int t = 32 * qw + lane;               // this thread's token; its dim at the end
        const uint32_t tl = (uint32_t)(32 * qw) << 16;
        float *red = reinterpret_cast<float *>(smem + CC::OFF_RED);   // [4][32] stage maxima
        float *red2 = red + 4 * CC::N;                                 // [4][32] row sums
        float mref[8], lsum[8];
        int g = 0;
        for (int n = 0;; ++n) {
            const int b = n & 1;
            const bool okm = wait(CC::B_RECFULL + b, (uint32_t)((n >> 1) & 1));
            if (softmax_any(!okm))
                break;
            int32_t *m = meta(b);
            if (m[CC::M_END])
                break;
            const int32_t *it = rec_of(m);
            const int n_st = m[CC::M_NST], kvh = m[CC::M_KVH];
            const int nseg = it[plan::I_NSEG], total = it[plan::I_TILES], nrows = it[plan::I_NROWS];
            auto seg = [&](int k) { return it + CC::SEGS + plan::kSegInts * k; };
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                mref[i] = -INFINITY;
                lsum[i] = 0.f;
            }
            int kcur = 0;
            bool fail = false;
            for (int s = 0; s < n_st; ++s, ++g) {
                const int slot = g % NSTAGE, sb = g & 1;
                const bool oks = wait_poll(CC::B_SFULL + sb, (uint32_t)((g >> 1) & 1));
                if (softmax_any(!oks || aborted())) {
                    fail = true;
                    break;
                }
                tc05::fence_after_sync();
                uint32_t sv[8], sv2[8];
                tc05::ld8(tS + sb * 64 + r0 + tl, sv);
                tc05::ld8(tS + sb * 64 + 32 + r0 + tl, sv2);
                tc05::wait_ld();
                tc05::fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&bars[CC::B_SFREE + sb]);   // the score buffer may take stage g + 2

                // this token's place: tile, segment, rows it serves
                const int tile = TPS * s + t / TILE;
                const bool loaded = tile < total;
                bool valid = false;
                int rlo = 0, rhi = 0;
                if (loaded) {
                    while (kcur + 1 < nseg && seg(kcur + 1)[plan::S_FIRST_TILE] <= tile)
                        ++kcur;
                    const int *gg = seg(kcur);
                    const int tok = gg[plan::S_BEGIN] + (tile - gg[plan::S_FIRST_TILE]) * TILE + t % TILE;
                    valid = tok < gg[plan::S_END];
                    rlo = gg[plan::S_ROW_LO];
                    rhi = min(gg[plan::S_ROW_HI], nrows);
                }
                float x[8];
                bool over = false;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const bool live = valid && r0 + i >= rlo && r0 + i < rhi;
                    x[i] = live ? (__uint_as_float(sv[i]) + __uint_as_float(sv2[i])) * p.qscale : -INFINITY;
                    over |= x[i] > mref[i] + kSlack;   // a row with no token yet: any live score
                }
                if (softmax_any(over)) {
                    // exact maxima of this stage's scores per row: over the
                    // warp's 32 tokens, then over the four lane quarters
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        float v = x[i];
                        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
                        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
                        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
                        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
                        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
                        if (lane == i)
                            red[qw * CC::N + r0 + i] = v;
                    }
                    softmax_sync();
                    float alpha[8];
                    bool grew = false;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int r = r0 + i;
                        const float sm = fmaxf(fmaxf(red[r], red[CC::N + r]),
                                               fmaxf(red[2 * CC::N + r], red[3 * CC::N + r]));
                        const float mn = fmaxf(mref[i], sm);
                        // a row with no token so far keeps nothing to rescale
                        alpha[i] = mn == -INFINITY ? 1.f : fast_exp2(mref[i] - mn);
                        grew |= mn != mref[i];
                        mref[i] = mn;
                    }
                    bool okr = true;
                    if (grew && s > 0) {
                        // O holds this item's earlier stages: rescale this row
                        // group's columns once their products are done
                        okr = wait(CC::B_STFREE + (g - 1) % NSTAGE, (uint32_t)(((g - 1) / NSTAGE) & 1));
                        if (okr) {
                            tc05::fence_after_sync();
                            uint32_t ov[4][8];   // (even, odd tile) x (hi, lo) columns of the group's rows
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                tc05::ld8(tO + 32 * q + r0 + tl, ov[q]);
                            tc05::wait_ld();
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
#pragma unroll
                                for (int i = 0; i < 8; ++i)
                                    ov[q][i] = __float_as_uint(__uint_as_float(ov[q][i]) * alpha[i]);
                                tc05::st8(tO + 32 * q + r0 + tl, ov[q]);
                            }
                            tc05::wait_st();
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        lsum[i] *= alpha[i];
                    if (softmax_any(!okr)) {
                        fail = true;
                        break;
                    }
                }
                // P = hi + lo: this token's 8 rows of the B operand [token][rows]
                // over the stage's K, one 16-byte piece (the row group's),
                // swizzled by the token's row within its 8-token atom
                uint8_t *kb = smem + slot * CC::STAGE;
                {
                    uint32_t h[4], lo[4];
#pragma unroll
                    for (int w2 = 0; w2 < 4; ++w2) {
                        const float a0 = x[2 * w2] == -INFINITY ? 0.f : fast_exp2(x[2 * w2] - mref[2 * w2]);
                        const float a1 = x[2 * w2 + 1] == -INFINITY ? 0.f
                                                                     : fast_exp2(x[2 * w2 + 1] - mref[2 * w2 + 1]);
                        lsum[2 * w2] += a0;
                        lsum[2 * w2 + 1] += a1;
                        h[w2] = Mma<T>::pack(a0, a1);
                        const float2 hf = Mma<T>::unpack(h[w2]);
                        lo[w2] = Mma<T>::pack(a0 - hf.x, a1 - hf.y);
                    }
                    const uint32_t row = smem_u32(kb) + (uint32_t)((t >> 3) * 1024 + (t & 7) * 128);
                    const uint32_t ah = row + (uint32_t)(((j ^ (t & 7)) & 7) << 4);
                    const uint32_t al = row + (uint32_t)((((4 + j) ^ (t & 7)) & 7) << 4);
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(ah), "r"(h[0]), "r"(h[1]),
                                 "r"(h[2]), "r"(h[3])
                                 : "memory");
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(al), "r"(lo[0]),
                                 "r"(lo[1]), "r"(lo[2]), "r"(lo[3])
                                 : "memory");
                }
                // a loaded tile's rows past its segment may hold anything (even
                // NaN patterns): row group 0 zeroes such a token's V row so that
                // 0 * v stays 0
                if (j == 0 && loaded && !valid) {
                    if (wait(CC::B_VFULL + slot, (uint32_t)((g / NSTAGE) & 1))) {
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            uint4 *vr = reinterpret_cast<uint4 *>(kb + CC::KV_BYTES + c * CC::PLANE + t * 128);
#pragma unroll
                            for (int q8 = 0; q8 < 8; ++q8)   // pieces staggered across the rows' banks
                                vr[(q8 ^ t) & 7] = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                }
                fence_proxy_async_smem();   // P and the zeroed rows before the MMAs read them
                tc05::fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&bars[CC::B_PFULL + slot]);
            }
            if (fail)
                break;

            // ---- end of the item: row sums, O^T, outputs or partials (the
            // loader's check results are needed from here on)
            {
                bool oke = wait(CC::B_METAFULL + b, (uint32_t)((n >> 1) & 1));
                if (n_st > 0)
                    oke = oke && wait(CC::B_STFREE + (g - 1) % NSTAGE, (uint32_t)(((g - 1) / NSTAGE) & 1));
                if (softmax_any(!oke))
                    break;
                if (n_st > 0)
                    tc05::fence_after_sync();
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float v = lsum[i];
                v += __shfl_xor_sync(0xffffffffu, v, 16);
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                if (lane == i)
                    red2[qw * CC::N + r0 + i] = v;
            }
            float ov[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                ov[i] = 0.f;
            if (n_st > 0) {
                // the four partial sums; the odd-tile ones hold nothing of an
                // item with a single tile
                uint32_t o4[4][8];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    tc05::ld8(tO + 32 * q + r0 + tl, o4[q]);
                tc05::wait_ld();
                const bool odd = total > 1;
#pragma unroll
                for (int i = 0; i < 8; ++i)   // (even hi + even lo) + (odd hi + odd lo)
                    ov[i] = (__uint_as_float(o4[0][i]) + __uint_as_float(o4[1][i])) +
                            (odd ? __uint_as_float(o4[2][i]) + __uint_as_float(o4[3][i]) : 0.f);
            }
            tc05::fence_before_sync();
            softmax_sync();
            const int32_t *members = it + plan::kItemHead;
            const CtaWork w{it[plan::I_SEQ0], nrows, kvh, 0, 0, it[plan::I_SLOT], it[plan::I_SEQ0], members};
            const uint32_t badrows = (uint32_t)m[CC::M_BADROWS], fin = (uint32_t)m[CC::M_FINAL];
            const bool zero = m[CC::M_ZERO] != 0, failed_all = m[CC::M_FAILED] != 0;
            const int rows = nrows > 0 && nrows <= RQ ? nrows : 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = r0 + i;
                if (r < rows) {
                    const float L = (red2[r] + red2[CC::N + r]) + (red2[2 * CC::N + r] + red2[3 * CC::N + r]);
                    const int64_t sh = row_head(p, w, G, r);
                    const bool bad = failed_all || ((badrows >> r) & 1u);
                    const float o = ov[i];
                    if ((fin >> r) & 1u) {
                        store_out(p.out, p.out_dtype, sh * D + t,
                                  (zero || bad || !(L > 0.f)) ? 0.f : o * (1.f / L));
                    } else {
                        const int64_t base = sh * slots + it[plan::I_SLOT];
                        __stcg(p.ws_acc + base * D + t, bad ? 0.f : o);
                        if (t == 0)
                            __stcg(reinterpret_cast<float2 *>(p.ws_ml) + base,
                                   make_float2(bad ? -INFINITY : mref[i], bad ? -1.f : L));
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars[CC::B_RECEMPTY + b]);
        }
    }

    // every warp's last access to the tensor memory precedes its arrival
    // here; the allocating warp frees it once all have arrived (no CTA-wide
    // barrier: the roles' lane 0 threads reconverge with their warps first)
    __syncwarp();
    tc05::fence_before_sync();
    if (lane == 0)
        mbar_arrive(&bars[CC::B_DONE]);
    if (warp == 1) {
        drain_wait(&bars[CC::B_DONE], 0u, p.status);
        tc05::fence_after_sync();
        tc05::dealloc(tS, CC::TM_COLS);
    }
}

}  // namespace pkv
