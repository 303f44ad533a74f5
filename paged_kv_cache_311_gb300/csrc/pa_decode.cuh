// pa_decode.cuh -- paged decode attention for sm_103a.
//
// What it computes (PagedAttention: Efficient LLM Serving with vLLM, "The
// PagedAttention Algorithm", Steps 4-5): for every sequence s and query head
// h, the softmax(scale * q[s,h] . k_i)-weighted sum of v_i over the
// sequence's logical tokens i < L_s, where token i lives in physical block
// block_tables[s][i / bs], row i % bs, of a cache laid out [num_blocks, Hk,
// bs, D].
//
// Kernel design (one CTA per (context partition, kv head, sequence)):
//   * The CTA owns the G = H / Hk query heads of one kv head, so every K/V
//     byte is read from HBM once and feeds G heads.
//   * Each warp streams its own tiles of 16 tokens through an S-stage ring in
//     shared memory.  Lane 0 of the warp is the producer: per tile it issues
//     one TMA load (cp.async.bulk.tensor.5d) per block-box of K and of V,
//     completing on the stage's mbarrier.  The tensor map writes each box as
//     [128-byte chunk][row][128 bytes] with 128-byte swizzling, which makes
//     both token-major and dim-major shared-memory reads conflict-free.
//     Block ids come from the partition's slice of the block table, staged in
//     shared memory when the CTA starts.
//   * Two interchangeable per-warp engines consume a tile:
//       CcEngine (CUDA cores): QK with two lanes per token and q broadcast
//         from shared memory, PV with D/32 dims of all G heads per lane,
//         packed fp32x2 FMAs; for fp32 caches and small G.
//       TcEngine (tensor cores, mma.sync m16n8k16): for 16-bit caches, the
//         tile is the M = 16 dimension and the (up to 8) query heads the
//         N = 8 dimension: S^T = K q^T from ldmatrix'd K, O^T += V^T P^T with
//         ldmatrix.trans'd V and P^T transposed in registers (movmatrix).  P
//         is split into a 16-bit high part and a 16-bit remainder so that the
//         products keep fp32-level accuracy; accumulation is fp32.
//     Both run the online softmax per tile in the log2 domain (exp2).
//   * End of CTA: warps merge (max, sum, acc) through shared memory; the
//     single-pass kernel writes the normalised output, the split-context
//     kernel writes (max, sum, unnormalised acc) to the workspace for the
//     log-sum-exp reduce kernel.
//   * Reduction order depends only on logical token positions, so results
//     are bit-identical under any physical placement of the blocks.
#pragma once

#include <type_traits>

#include "pkv_device.cuh"

namespace pkv {

struct DecodeParams {
    void *out;
    const void *q;
    const int32_t *block_tables;
    const int32_t *context_lens;
    float *ws_ml;     // split path: [B][H][NP][2] = (max, sum) in the log2 domain
    float *ws_acc;    // split path: [B][H][NP][D] unnormalised accumulators
    uint32_t *status;
    int64_t num_blocks;
    int num_seqs, num_heads, num_kv_heads;
    int max_blocks_per_seq;
    int max_context_len;
    int partition_size;  // tokens per CTA along the context
    int num_partitions;  // grid.x
    int out_dtype;
    int split;           // nonzero: write partials to the workspace
    float qscale;        // softmax scale * log2(e)
    int num_items;       // shared-prefix plans: work items in the plan
};

enum Engine { kEngineAuto = 0, kEngineCudaCore = 1, kEngineTensorCore = 2, kEngineTcgen05 = 3 };

#ifndef PKV_DECODE_STAGE_BUDGET_CC
#define PKV_DECODE_STAGE_BUDGET_CC 98304
#endif
#ifndef PKV_DECODE_STAGE_BUDGET_TC
#define PKV_DECODE_STAGE_BUDGET_TC 65536
#endif

template <typename T, int D, int BS, int G, bool TC>
struct DecodeCfg {
    static constexpr int E = Elem<T>::bytes;
    static constexpr int TILE = 16;                // tokens per warp tile
    static constexpr int NW = 4;                   // warps per CTA
    static constexpr int ROW = D * E;              // bytes of one token row
    static constexpr int CHUNKS = ROW / 128;       // 128-byte swizzle atoms per row
    static constexpr int EPP = 16 / E;             // elements per 16-byte piece
    static constexpr int NPC = ROW / 16;           // pieces per row
    static constexpr int BOX_ROWS = BS < TILE ? BS : TILE;
    static constexpr int BOXES = TILE / BOX_ROWS;
    static constexpr int BOX_BYTES = BOX_ROWS * ROW;
    static constexpr int TILE_BYTES = TILE * ROW;  // K (or V) of one tile
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int BUDGET = TC ? PKV_DECODE_STAGE_BUDGET_TC : PKV_DECODE_STAGE_BUDGET_CC;
    static constexpr int S0 = BUDGET / (NW * STAGE_BYTES);
    static constexpr int S = S0 < 2 ? 2 : (S0 > 8 ? 8 : S0);  // ring depth per warp
    static constexpr int TABLE_CAP = 1024;         // block-table entries per CTA
    // CUDA-core engine: shared-memory q (padded rows) and (p, p) pairs.
    static constexpr int QROW = G * EPP * 4 + 16;
    static constexpr int Q_BYTES = TC ? 0 : ((NPC * QROW + 127) / 128) * 128;
    static constexpr int P_BYTES = TC ? 0 : NW * TILE * G * 8;

    static constexpr int OFF_STAGES = 0;
    static constexpr int STAGES_BYTES = NW * S * STAGE_BYTES;
    static constexpr int OFF_Q = STAGES_BYTES;
    static constexpr int OFF_P = OFF_Q + Q_BYTES;
    static constexpr int OFF_TABLE = OFF_P + P_BYTES;
    static constexpr int OFF_BAR = OFF_TABLE + TABLE_CAP * 4;
    static constexpr int OFF_FLAG = OFF_BAR + NW * S * 8;
    static constexpr int SMEM_USED = OFF_FLAG + 16;
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack for 1024-byte alignment

    static_assert(ROW % 128 == 0, "rows must be whole 128-byte swizzle atoms");
    static_assert(TILE % BOX_ROWS == 0 && BOX_ROWS % 8 == 0, "box rows");
    static_assert(BOX_BYTES % 1024 == 0, "TMA 128B-swizzle boxes need 1024-byte alignment");
    static_assert(D % 64 == 0, "head_dim");
    static_assert(!TC || (E == 2 && G <= 8), "tensor-core engine: 16-bit caches, G <= 8");
    static_assert(NW * G * (D + 2) * 4 <= STAGES_BYTES, "merge scratch fits in the ring");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");

    // Shared-memory address of 16-byte piece `q` of token row `t` of a tile.
    __device__ __forceinline__ static uint32_t addr(uint32_t base, int t, int q)
    {
        const int bx = t / BOX_ROWS, r = t % BOX_ROWS;
        return base + bx * BOX_BYTES + ((q >> 3) * BOX_ROWS + r) * 128 + (((q & 7) ^ (r & 7)) << 4);
    }
};

// Host-visible description of the config (for the TMA box and launch).
template <typename T, int D, int BS, int G, bool TC>
struct DecodeShape {
    using C = DecodeCfg<T, D, BS, G, TC>;
    static constexpr int box_rows = C::BOX_ROWS;
    static constexpr int threads = C::NW * 32;
    static constexpr int smem = C::SMEM_BYTES;
};

__device__ __forceinline__ void store_out(void *out, int dtype, int64_t i, float v)
{
    if (dtype == PKV_F32)
        static_cast<float *>(out)[i] = v;
    else if (dtype == PKV_F16)
        static_cast<__half *>(out)[i] = __float2half_rn(v);
    else
        static_cast<__nv_bfloat16 *>(out)[i] = __float2bfloat16_rn(v);
}

// Four consecutive outputs from element i (a multiple of 4; the output is
// 16-byte aligned): one 16- or 8-byte store.
__device__ __forceinline__ void store_out4(void *out, int dtype, int64_t i, float4 v)
{
    if (dtype == PKV_F32) {
        *reinterpret_cast<float4 *>(static_cast<float *>(out) + i) = v;
    } else if (dtype == PKV_F16) {
        const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
        *reinterpret_cast<uint2 *>(static_cast<__half *>(out) + i) =
            make_uint2(*reinterpret_cast<const uint32_t *>(&a), *reinterpret_cast<const uint32_t *>(&b));
    } else {
        const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
        *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(out) + i) =
            make_uint2(*reinterpret_cast<const uint32_t *>(&a), *reinterpret_cast<const uint32_t *>(&b));
    }
}

// What one CTA computes: query rows r < nrows, row r being head
// (kvh * G + r % G) of sequence seq0 + r / G, over the tokens [tok0, tok_end)
// that the block table of `table_seq` addresses; split partials go to
// workspace slot `slot`.
// Query rows r < nrows of a CTA are head r % G (of its kv head's group) of
// sequence seq0 + r / G, or of members[r / G] when the CTA serves an explicit
// list of sequences (a shared-prefix item).
struct CtaWork {
    int seq0, nrows, kvh, tok0, tok_end, slot, table_seq;
    const int32_t *members = nullptr;
};

__device__ __forceinline__ int64_t row_head(const DecodeParams &p, const CtaWork &w, int G, int r)
{
    const int seq = w.members ? w.members[r / G] : w.seq0 + r / G;
    return (int64_t)seq * p.num_heads + w.kvh * G + r % G;
}

// Writes the result of a CTA that cannot produce one (bad length / block):
// zeros for the single pass, an "invalid" (max = -inf, sum = -1) marker for
// the split path.
template <int D, int G>
__device__ void write_invalid(const DecodeParams &p, const CtaWork &w)
{
    for (int idx = threadIdx.x; idx < w.nrows * D; idx += blockDim.x) {
        const int r = idx / D, d = idx % D;
        const int64_t sh = row_head(p, w, G, r);
        if (!p.split) {
            store_out(p.out, p.out_dtype, sh * D + d, 0.f);
        } else {
            const int64_t slot = sh * p.num_partitions + w.slot;
            p.ws_acc[slot * D + d] = 0.f;
            if (d == 0) {
                p.ws_ml[slot * 2 + 0] = -INFINITY;
                p.ws_ml[slot * 2 + 1] = -1.f;
            }
        }
    }
}

// ------------------------------------------------------------ CUDA cores
template <typename T, int D, int BS, int G>
struct CcEngine {
    using C = DecodeCfg<T, D, BS, G, false>;
    static constexpr int LPT = 32 / C::TILE;   // lanes per token in QK
    static constexpr int PCL = 8 / LPT;        // pieces per 128-byte chunk per lane
    static constexpr int DPL = D / 32;         // PV dims per lane
    static constexpr int VBYTES = DPL * C::E;  // PV bytes per lane per row
    static constexpr int AWS = D;              // accumulator row stride of the merge scratch

    float m[G], lsum[G];
    float2 acc[G][DPL / 2];
    uint32_t qbase, pbase;
    int ti, sub, vq, vin;

    // Stages q (pre-scaled by scale * log2 e) as [piece][head][EPP] fp32.
    __device__ static void stage_q(const DecodeParams &p, uint8_t *smem, int seq, int kvh)
    {
        const T *qp = static_cast<const T *>(p.q) + ((int64_t)seq * p.num_heads + kvh * G) * D;
        for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
            const int h = i / D, d = i % D;
            float *dst = reinterpret_cast<float *>(smem + C::OFF_Q + (d / C::EPP) * C::QROW);
            dst[h * C::EPP + d % C::EPP] = to_float(qp[i]) * p.qscale;
        }
    }

    __device__ void init(const DecodeParams &, uint8_t *smem, const CtaWork &, int warp, int lane)
    {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            m[h] = -INFINITY;
            lsum[h] = 0.f;
#pragma unroll
            for (int k = 0; k < DPL / 2; ++k)
                acc[h][k] = make_float2(0.f, 0.f);
        }
        ti = lane / LPT;
        sub = lane % LPT;
        qbase = smem_u32(smem + C::OFF_Q);
        pbase = smem_u32(smem + C::OFF_P) + warp * C::TILE * G * 8;
        vq = (lane * VBYTES) >> 4;
        vin = (lane * VBYTES) & 15;
    }

    __device__ void tile(uint32_t kbase, uint32_t vbase, int nvalid, int lane)
    {
        // ---- QK for token ti
        float2 s2[G];
#pragma unroll
        for (int h = 0; h < G; ++h)
            s2[h] = make_float2(0.f, 0.f);
#pragma unroll
        for (int c2 = 0; c2 < C::CHUNKS; ++c2) {
#pragma unroll
            for (int i4 = 0; i4 < PCL; ++i4) {
                const int pc = sub * PCL + i4;
                const uint4 kw = lds128(C::addr(kbase, ti, c2 * 8 + pc));
                const uint32_t qa = qbase + (c2 * 8 + pc) * C::QROW;
                if constexpr (C::E == 2) {
                    const float2 k0 = Unpack<T>::pair(kw.x), k1 = Unpack<T>::pair(kw.y);
                    const float2 k2 = Unpack<T>::pair(kw.z), k3 = Unpack<T>::pair(kw.w);
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const float4 qa0 = lds128f(qa + h * 32);
                        const float4 qa1 = lds128f(qa + h * 32 + 16);
                        s2[h] = ffma2(make_float2(qa0.x, qa0.y), k0, s2[h]);
                        s2[h] = ffma2(make_float2(qa0.z, qa0.w), k1, s2[h]);
                        s2[h] = ffma2(make_float2(qa1.x, qa1.y), k2, s2[h]);
                        s2[h] = ffma2(make_float2(qa1.z, qa1.w), k3, s2[h]);
                    }
                } else {
                    const float2 k0 = make_float2(__uint_as_float(kw.x), __uint_as_float(kw.y));
                    const float2 k1 = make_float2(__uint_as_float(kw.z), __uint_as_float(kw.w));
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const float4 qa0 = lds128f(qa + h * 16);
                        s2[h] = ffma2(make_float2(qa0.x, qa0.y), k0, s2[h]);
                        s2[h] = ffma2(make_float2(qa0.z, qa0.w), k1, s2[h]);
                    }
                }
            }
        }

        // ---- online softmax over this tile (log2 domain)
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float s = s2[h].x + s2[h].y;
#pragma unroll
            for (int off = 1; off < LPT; off <<= 1)
                s += __shfl_xor_sync(0xffffffffu, s, off);
            s = ti < nvalid ? s : -INFINITY;
            float tm = s;
#pragma unroll
            for (int off = LPT; off < 32; off <<= 1)
                tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, off));
            const float mn = fmaxf(m[h], tm);
            const float alpha = exp2f(m[h] - mn);
            const float pr = exp2f(s - mn);
            lsum[h] = lsum[h] * alpha + (sub == 0 ? pr : 0.f);
            const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
            for (int k = 0; k < DPL / 2; ++k)
                acc[h][k] = fmul2(acc[h][k], a2);
            m[h] = mn;
            if (sub == 0)
                asm volatile("st.shared.v2.f32 [%0], {%1, %1};" ::"r"(pbase + (ti * G + h) * 8),
                             "f"(pr)
                             : "memory");
        }
        __syncwarp();

        // ---- PV: this lane's D/32 dims of every head
        for (int t = 0; t < nvalid; ++t) {
            const uint32_t va = C::addr(vbase, t, vq) + vin;
            float2 vf[DPL / 2];
            if constexpr (C::E == 2) {
                if constexpr (VBYTES == 8) {
                    const uint2 w = lds64(va);
                    vf[0] = Unpack<T>::pair(w.x);
                    vf[1] = Unpack<T>::pair(w.y);
                } else {
                    vf[0] = Unpack<T>::pair(lds32(va));
                }
            } else {
                if constexpr (VBYTES == 16) {
                    const float4 w = lds128f(va);
                    vf[0] = make_float2(w.x, w.y);
                    vf[1] = make_float2(w.z, w.w);
                } else {
                    vf[0] = lds64f(va);
                }
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float2 pp = lds64f(pbase + (t * G + h) * 8);
#pragma unroll
                for (int k = 0; k < DPL / 2; ++k)
                    acc[h][k] = ffma2(pp, vf[k], acc[h][k]);
            }
        }
    }

    // Per-warp (max, sum, acc) of every head into the merge scratch (rows
    // are the G heads, row stride G).
    __device__ void finish(float *mw, float *lw, float *aw, int warp, int lane, int)
    {
#pragma unroll
        for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                lsum[h] += __shfl_xor_sync(0xffffffffu, lsum[h], off);
        }
        if (lane == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                mw[warp * G + h] = m[h];
                lw[warp * G + h] = lsum[h];
            }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int k = 0; k < DPL / 2; ++k)
                *reinterpret_cast<float2 *>(&aw[(warp * G + h) * D + lane * DPL + 2 * k]) = acc[h][k];
        }
    }
};

// 2^x on the special-function unit (ex2.approx.ftz: relative error near
// 2^-22, subnormal results flushed to zero), for the probabilities of the
// tensor-core engine: each is at most 2^8 and is split into 16-bit high and
// low parts that keep 16 bits of it, far coarser than that error.
__device__ __forceinline__ float ex2_fast(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------- tensor cores
// NT n-tiles of 8 query rows each (NT = 1 for one sequence's G <= 8 heads).
// QS: the q^T B-fragments are read from a shared-memory copy of the rows
// (q_smem_bytes, staged by the caller before init) with ldmatrix at every
// tile instead of being held in registers -- 16 * NT registers fewer, for
// the multi-row (shared-prefix) CTAs.
template <typename T, int D, int BS, int G, int NT = 1, bool QS = false>
struct TcEngine {
    using C = DecodeCfg<T, D, BS, G, true>;
    static constexpr int KS = D / 16;   // k-steps of QK = m-tiles of PV
    static constexpr int RS = 8 * NT;   // row stride of the merge scratch
    // accumulator row stride of the merge scratch, in floats: padded so that
    // the rows 2c, 2c + 1 of one store fall in distinct banks
    static constexpr int AWS = D + 4;
    // shared-memory q rows: D 16-bit values padded by 16 bytes, so the 8
    // row addresses of one ldmatrix fall in distinct bank groups
    static constexpr int QROWB = D * 2 + 16;
    static constexpr int q_smem_bytes = RS * QROWB;

    uint32_t qf[QS ? 1 : KS][NT][2];   // q^T B-fragments: row 8 nt + g, dims 16 ks + 2c (+8)
    uint32_t qaddr;                    // QS: this lane's ldmatrix row address
    float o[KS][NT][4];       // O^T C-fragments: dims 16 mt + g (+8), rows 8 nt + 2c, +1
    float m[NT][2], lsum[NT][2];
    float qscale;
    int g, c, ntl;            // ntl: n-tiles that hold live rows
    // This lane's ldmatrix row offsets inside a tile (swizzle included): the
    // K matrices of k-step ks and the V matrices of m-tile mt, for ks, mt < 8
    // (the second 128-byte chunk adds a constant).
    uint32_t koff[4], voff[4];

    __device__ static void stage_q(const DecodeParams &, uint8_t *, int, int) {}

    // Chunk offset of k-step / m-tile k (its 16-byte pieces are 2k and 2k+1).
    __device__ __forceinline__ static uint32_t chunk_off(int k)
    {
        return (uint32_t)((k >> 2) * C::BOX_ROWS * 128);
    }

    // The CTA's query rows (rows >= nrows zero) on their way to shared memory
    // for QS engines, in two halves so that a caller can put other loads in
    // flight between them: load() issues every global load, store() writes
    // the rows at `qs`.  All C::NW * 32 threads of the CTA take part, and a
    // barrier must follow the stores before init.
    struct QRows {
        static constexpr int PCS = D * 2 / 16;   // 16-byte pieces per row
        static constexpr int PER = (RS * PCS + C::NW * 32 - 1) / (C::NW * 32);
        uint4 v[PER];

        __device__ __forceinline__ void load(const DecodeParams &p, const CtaWork &w)
        {
#pragma unroll
            for (int u = 0; u < PER; ++u) {
                const int i = threadIdx.x + u * C::NW * 32, r = i / PCS;
                v[u] = make_uint4(0u, 0u, 0u, 0u);
                if (i < RS * PCS && r < w.nrows)
                    v[u] = reinterpret_cast<const uint4 *>(static_cast<const T *>(p.q) +
                                                           row_head(p, w, G, r) * D)[i % PCS];
            }
        }
        __device__ __forceinline__ void store(uint8_t *qs) const
        {
#pragma unroll
            for (int u = 0; u < PER; ++u) {
                const int i = threadIdx.x + u * C::NW * 32;
                if (i < RS * PCS)
                    *reinterpret_cast<uint4 *>(qs + (i / PCS) * QROWB + (i % PCS) * 16) = v[u];
            }
        }
    };

    __device__ void init(const DecodeParams &p, uint8_t *qs, const CtaWork &w, int, int lane)
    {
        g = lane >> 2;
        c = lane & 3;
        qscale = p.qscale;
        ntl = (w.nrows + 7) / 8;
        if constexpr (QS)
            qaddr = smem_u32(qs) + (lane & 7) * QROWB + (lane >> 3) * 16;
        {
            const int tk = (lane & 7) + ((lane >> 3) & 1) * 8, dk = lane >> 4;
            const int tv = (lane & 7) + (lane >> 4) * 8, dv = (lane >> 3) & 1;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                koff[k] = C::addr(0, tk, 2 * k + dk);
                voff[k] = C::addr(0, tv, 2 * k + dv);
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int r = 8 * nt + g;
            const bool live = r < w.nrows;
            const uint32_t *qp = reinterpret_cast<const uint32_t *>(
                static_cast<const T *>(p.q) + row_head(p, w, G, live ? r : 0) * D);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                if constexpr (!QS) {
                    qf[ks][nt][0] = live ? qp[(16 * ks + 2 * c) / 2] : 0u;
                    qf[ks][nt][1] = live ? qp[(16 * ks + 2 * c + 8) / 2] : 0u;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    o[ks][nt][j] = 0.f;
            }
            m[nt][0] = m[nt][1] = -INFINITY;
            lsum[nt][0] = lsum[nt][1] = 0.f;
        }
    }

    // Rows outside [row_lo, row_hi) ignore the tile (their state is unchanged):
    // only the n-tiles holding such rows run, each range of them in its own
    // straight-line copy of the tile (a tail tile of one member costs one
    // n-tile's MMAs and softmax, not NT's).
    __device__ void tile(uint32_t kbase, uint32_t vbase, int nvalid, int lane, int row_lo = 0,
                         int row_hi = 1 << 30)
    {
        const int nlo = row_lo >> 3, nhi = min(ntl, (row_hi + 7) >> 3);
        if constexpr (NT == 1) {
            if (nhi > nlo)
                tile_rows<0, 1>(kbase, vbase, nvalid, lane, row_lo, row_hi);
        } else {
            static_assert(NT == 3, "n-tile ranges are dispatched for NT = 1 and 3");
            switch (nlo * 4 + nhi) {
            case 0 * 4 + 3: tile_rows<0, 3>(kbase, vbase, nvalid, lane, row_lo, row_hi); break;
            case 0 * 4 + 1: tile_rows<0, 1>(kbase, vbase, nvalid, lane, row_lo, row_hi); break;
            case 1 * 4 + 2: tile_rows<1, 2>(kbase, vbase, nvalid, lane, row_lo, row_hi); break;
            case 2 * 4 + 3: tile_rows<2, 3>(kbase, vbase, nvalid, lane, row_lo, row_hi); break;
            case 0 * 4 + 2: tile_rows<0, 2>(kbase, vbase, nvalid, lane, row_lo, row_hi); break;
            case 1 * 4 + 3: tile_rows<1, 3>(kbase, vbase, nvalid, lane, row_lo, row_hi); break;
            default: break;   // no n-tile holds a row of the tile
            }
        }
    }

    // The tile over n-tiles [N0, N1).
    template <int N0, int N1>
    __device__ __forceinline__ void tile_rows(uint32_t kbase, uint32_t vbase, int nvalid, int lane,
                                              int row_lo, int row_hi)
    {
        // ---- S^T (16 tokens x 8 query rows per n-tile) = K q^T, as two
        // independent accumulation chains (even / odd k-steps)
        float s[NT][4], s2[NT][4];
#pragma unroll
        for (int nt = N0; nt < N1; ++nt)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                s[nt][j] = s2[nt][j] = 0.f;
        if constexpr (QS) {
            // one ldmatrix.x4 of q gives the fragments of k-steps 2 kp, 2 kp + 1;
            // with several n-tiles, their chains are the independent ones
#pragma unroll
            for (int kp = 0; kp < KS / 2; ++kp) {
                uint32_t a0[4], a1[4];
                ldsm_x4(kbase + chunk_off(2 * kp) + koff[(2 * kp) & 3], a0);
                ldsm_x4(kbase + chunk_off(2 * kp + 1) + koff[(2 * kp + 1) & 3], a1);
#pragma unroll
                for (int nt = N0; nt < N1; ++nt) {
                        uint32_t b[4];
                        ldsm_x4(qaddr + nt * 8 * QROWB + kp * 64, b);
                        Mma<T>::run(s[nt], a0, b[0], b[1]);
                        Mma<T>::run(NT > 1 ? s[nt] : s2[nt], a1, b[2], b[3]);
                    }
            }
        } else {
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                uint32_t a[4];
                ldsm_x4(kbase + chunk_off(ks) + koff[ks & 3], a);
#pragma unroll
                for (int nt = N0; nt < N1; ++nt) {
                        if (ks & 1)
                            Mma<T>::run(s2[nt], a, qf[ks][nt][0], qf[ks][nt][1]);
                        else
                            Mma<T>::run(s[nt], a, qf[ks][nt][0], qf[ks][nt][1]);
                    }
            }
        }
        if constexpr (NT == 1 || !QS) {   // QS with several n-tiles: one chain per n-tile
#pragma unroll
            for (int nt = N0; nt < N1; ++nt)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    s[nt][j] += s2[nt][j];
        }

        // ---- online softmax in the log2 domain: this lane holds tokens g,
        // g + 8 of rows 2c, 2c + 1.  Each row keeps a reference maximum m.
        // While every new score of the warp stays within kSlack of its row's
        // reference -- the common case once a row has seen a tile -- the
        // probabilities 2^(x - m) <= 2^kSlack are taken against the unchanged
        // reference: no cross-lane maximum, no rescale (fp32 sums and the
        // hi/lo 16-bit split of P lose nothing at that size).  Otherwise every
        // row moves to its exact running maximum and the accumulators are
        // rescaled.  (m, lsum, o) always share one reference, which is all the
        // merges need.
        constexpr float kSlack = 8.f;
        const bool ok0 = g < nvalid, ok1 = g + 8 < nvalid;
        float x0[NT][2], x1[NT][2], p0[NT][2], p1[NT][2];
        bool over = false;
#pragma unroll
        for (int nt = N0; nt < N1; ++nt) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int row = 8 * nt + 2 * c + j;
                const bool live = row >= row_lo && row < row_hi;
                x0[nt][j] = (ok0 && live) ? s[nt][j] * qscale : -INFINITY;
                x1[nt][j] = (ok1 && live) ? s[nt][2 + j] * qscale : -INFINITY;
                // a row with no token yet (m = -inf) is over for any live score
                over |= fmaxf(x0[nt][j], x1[nt][j]) > m[nt][j] + kSlack;
            }
        }
        if (!__any_sync(0xffffffffu, over)) {
#pragma unroll
            for (int nt = N0; nt < N1; ++nt) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    // rows still without a token have no live score here: the
                    // finite stand-in keeps 2^(-inf - m) at 0 instead of NaN
                    const float mr = fmaxf(m[nt][j], -1e30f);
                    p0[nt][j] = ex2_fast(x0[nt][j] - mr);
                    p1[nt][j] = ex2_fast(x1[nt][j] - mr);
                    lsum[nt][j] += p0[nt][j] + p1[nt][j];
                }
            }
        } else {
            float alpha[NT][2];
            bool grew = false;
#pragma unroll
            for (int nt = N0; nt < N1; ++nt) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    float tm = fmaxf(x0[nt][j], x1[nt][j]);
                    tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 4));
                    tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 8));
                    tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 16));
                    const float mn = fmaxf(m[nt][j], tm);
                    // a row with no token yet keeps max -inf: nothing to rescale or add
                    const bool none = mn == -INFINITY;
                    alpha[nt][j] = none ? 1.f : ex2_fast(m[nt][j] - mn);
                    grew |= mn != m[nt][j];
                    p0[nt][j] = none ? 0.f : ex2_fast(x0[nt][j] - mn);
                    p1[nt][j] = none ? 0.f : ex2_fast(x1[nt][j] - mn);
                    lsum[nt][j] = lsum[nt][j] * alpha[nt][j] + p0[nt][j] + p1[nt][j];
                    m[nt][j] = mn;
                }
            }
            // rescale the accumulators only when some row's running maximum moved
            if (__any_sync(0xffffffffu, grew)) {
#pragma unroll
                for (int nt = N0; nt < N1; ++nt)
#pragma unroll
                    for (int mt = 0; mt < KS; ++mt) {
                        o[mt][nt][0] *= alpha[nt][0];
                        o[mt][nt][1] *= alpha[nt][1];
                        o[mt][nt][2] *= alpha[nt][0];
                        o[mt][nt][3] *= alpha[nt][1];
                    }
            }
        }

        // ---- rows of V past the valid tokens may hold anything (even NaN
        // bit patterns); zero them so that 0 * v stays 0 in the PV products.
        if (nvalid < C::TILE) {
            for (int idx = lane; idx < (C::TILE - nvalid) * C::NPC; idx += 32) {
                const int t = nvalid + idx / C::NPC, q = idx % C::NPC;
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(C::addr(vbase, t, q)),
                             "r"(0u)
                             : "memory");
            }
            __syncwarp();
        }

        // ---- P^T B-fragments: P = hi + lo in the cache's 16-bit type
        uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
        for (int nt = N0; nt < N1; ++nt) {
            const uint32_t h0 = Mma<T>::pack(p0[nt][0], p0[nt][1]);  // tokens g,   rows 2c, 2c+1
            const uint32_t h1 = Mma<T>::pack(p1[nt][0], p1[nt][1]);  // tokens g+8, rows 2c, 2c+1
            const float2 f0 = Mma<T>::unpack(h0), f1 = Mma<T>::unpack(h1);
            const uint32_t l0 = Mma<T>::pack(p0[nt][0] - f0.x, p0[nt][1] - f0.y);
            const uint32_t l1 = Mma<T>::pack(p1[nt][0] - f1.x, p1[nt][1] - f1.y);
            bh[nt][0] = movmatrix_trans(h0);
            bh[nt][1] = movmatrix_trans(h1);
            bl[nt][0] = movmatrix_trans(l0);
            bl[nt][1] = movmatrix_trans(l1);
        }

        // ---- O^T (D dims x 8 rows per n-tile) += V^T P^T
        {
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                uint32_t a[4];
                ldsm_x4_trans(vbase + chunk_off(mt) + voff[mt & 3], a);
#pragma unroll
                for (int nt = N0; nt < N1; ++nt) {
                    Mma<T>::run(o[mt][nt], a, bh[nt][0], bh[nt][1]);
                    Mma<T>::run(o[mt][nt], a, bl[nt][0], bl[nt][1]);
                }
            }
        }
    }

    // Per-warp (max, sum, acc) of live rows r < nrows into the merge scratch
    // (row stride RS).
    __device__ void finish(float *mw, float *lw, float *aw, int warp, int lane, int nrows)
    {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float l = lsum[nt][j];
                l += __shfl_xor_sync(0xffffffffu, l, 4);
                l += __shfl_xor_sync(0xffffffffu, l, 8);
                l += __shfl_xor_sync(0xffffffffu, l, 16);
                const int row = 8 * nt + 2 * c + j;
                if (row < nrows) {
                    if (g == 0) {
                        mw[warp * RS + row] = m[nt][j];
                        lw[warp * RS + row] = l;
                    }
#pragma unroll
                    for (int mt = 0; mt < KS; ++mt) {
                        aw[(warp * RS + row) * AWS + 16 * mt + g] = o[mt][nt][j];
                        aw[(warp * RS + row) * AWS + 16 * mt + g + 8] = o[mt][nt][2 + j];
                    }
                }
            }
        }
    }
};

// ------------------------------------------------------------ CTA body
// Initialises the per-warp ring barriers (once per CTA).
template <typename C>
__device__ __forceinline__ void init_rings(uint8_t *smem)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR) + warp * C::S;
        for (int s = 0; s < C::S; ++s)
            mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
}

// One CTA work unit: stage the block-table slice, stream the tiles through
// the per-warp rings, merge the warps and write the rows' output (single
// pass) or partials (split).  `ring` counts the tiles each warp has already
// pushed through its ring (stage and phase of the next tile follow from it);
// a CTA that runs several units passes the same counter to each.  Ends with
// a CTA barrier, so the next unit may reuse all shared memory.
template <typename T, int D, int BS, int G, bool TC, int NT>
__device__ __forceinline__ void decode_cta(const DecodeParams &p, const CUtensorMap *tmk,
                                           const CUtensorMap *tmv, uint8_t *smem, const CtaWork &w,
                                           int &ring)
{
    using C = DecodeCfg<T, D, BS, G, TC>;
    using Eng = typename std::conditional<TC, TcEngine<T, D, BS, G, NT>, CcEngine<T, D, BS, G>>::type;
    constexpr int NW = C::NW, S = C::S, TILE = C::TILE;
    constexpr int RS = TC ? 8 * NT : G;   // merge-scratch rows per warp
    static_assert(NW * RS * (Eng::AWS + 2) * 4 <= C::STAGES_BYTES, "merge scratch fits in the ring");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tok0 = w.tok0, tok_end = w.tok_end, kvh = w.kvh;

    // ---- stage the block-table slice (and, for the CUDA-core engine, q)
    const int j0 = tok0 / BS;
    const int nblk = (tok_end - tok0 + BS - 1) / BS;
    int32_t *table_s = reinterpret_cast<int32_t *>(smem + C::OFF_TABLE);
    const int32_t *bt = p.block_tables + (int64_t)w.table_seq * p.max_blocks_per_seq + j0;
    int bad = 0;
    for (int i = tid; i < nblk; i += NW * 32) {
        int b = bt[i];
        if (b < 0 || (int64_t)b >= p.num_blocks) {
            bad = 1;
            b = 0;
        }
        table_s[i] = b;
    }
    Eng::stage_q(p, smem, w.seq0, kvh);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR) + warp * S;
    uint32_t *cta_flag = reinterpret_cast<uint32_t *>(smem + C::OFF_FLAG);
    if (tid == 0) {
        *cta_flag = 0;
        prefetch_tensormap(tmk);
        prefetch_tensormap(tmv);
    }
    if (__syncthreads_or(bad)) {
        if (tid == 0)
            report(p.status, PKV_DEV_BAD_BLOCK);
        write_invalid<D, G>(p, w);
        __syncthreads();
        return;
    }

    // ---- per-warp tile stream
    const int ntok = tok_end - tok0;
    const int ntiles = (ntok + TILE - 1) / TILE;
    const int my_n = warp < ntiles ? (ntiles - 1 - warp) / NW + 1 : 0;
    uint8_t *stages = smem + C::OFF_STAGES + warp * S * C::STAGE_BYTES;

    const int base = ring;
    auto issue = [&](int i, int st) {
        const int t0 = tok0 + (warp + i * NW) * TILE;
        uint8_t *kd = stages + st * C::STAGE_BYTES;
        uint8_t *vd = kd + C::TILE_BYTES;
        const int nbox = min(C::BOXES, (tok_end - t0 + C::BOX_ROWS - 1) / C::BOX_ROWS);
        mbar_arrive_expect_tx(&bars[st], (uint32_t)(nbox * 2 * C::BOX_BYTES));
        for (int b = 0; b < nbox; ++b) {
            const int tok = t0 + b * C::BOX_ROWS;
            const int phys = table_s[tok / BS - j0];
            const int row0 = tok % BS;
            tma_load_5d(kd + b * C::BOX_BYTES, tmk, &bars[st], 0, row0, 0, kvh, phys);
            tma_load_5d(vd + b * C::BOX_BYTES, tmv, &bars[st], 0, row0, 0, kvh, phys);
        }
    };
    if (lane == 0) {
        const int pre = my_n < S ? my_n : S;
        if (pre > 0)
            fence_proxy_async_smem();  // a previous unit's merge wrote into the rings
        for (int i = 0; i < pre; ++i)
            issue(i, (base + i) % S);
    }

    Eng eng;
    eng.init(p, smem, w, warp, lane);

    int failed_at = -1;
    for (int i = 0; i < my_n; ++i) {
        const int st = (base + i) % S;
        if (!mbar_wait_bounded(&bars[st], (uint32_t)(((base + i) / S) & 1))) {
            failed_at = i;
            break;
        }
        const int t0 = tok0 + (warp + i * NW) * TILE;
        const int nvalid = min(TILE, tok_end - t0);
        const uint32_t kbase = smem_u32(stages + st * C::STAGE_BYTES);
        eng.tile(kbase, kbase + C::TILE_BYTES, nvalid, lane);
        __syncwarp();
        if (lane == 0 && i + S < my_n) {
            fence_proxy_async_smem();
            issue(i + S, st);
        }
    }

    if (failed_at >= 0) {
        // Drain the loads this warp still has in flight before the CTA may
        // exit, then mark the CTA's result invalid.
        const int last = min(my_n, failed_at + S);
        for (int i = failed_at; i < last; ++i)
            drain_wait(&bars[(base + i) % S], (uint32_t)(((base + i) / S) & 1), p.status);
        if (lane == 0) {
            report(p.status, PKV_DEV_TIMEOUT);
            atomicOr(cta_flag, 1u);
        }
    }

    ring = base + my_n;
    __syncthreads();  // every warp is done with its ring: reuse it as merge scratch
    const bool failed = *reinterpret_cast<volatile uint32_t *>(cta_flag) != 0;
    float *mw = reinterpret_cast<float *>(smem + C::OFF_STAGES);
    float *lw = mw + NW * RS;
    float *aw = lw + NW * RS;
    eng.finish(mw, lw, aw, warp, lane, w.nrows);
    __syncthreads();

    for (int idx = tid; idx < w.nrows * D; idx += NW * 32) {
        const int r = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int k = 0; k < NW; ++k)
            M = fmaxf(M, mw[k * RS + r]);
        float num = 0.f, den = 0.f;
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            const float mk = mw[k * RS + r];
            if (mk != -INFINITY) {
                const float f = exp2f(mk - M);
                num += f * aw[(k * RS + r) * Eng::AWS + d];
                den += f * lw[k * RS + r];
            }
        }
        const int64_t sh = row_head(p, w, G, r);
        if (!p.split) {
            store_out(p.out, p.out_dtype, sh * D + d, (failed || den == 0.f) ? 0.f : num / den);
        } else {
            const int64_t slot = sh * p.num_partitions + w.slot;
            p.ws_acc[slot * D + d] = failed ? 0.f : num;
            if (d == 0) {
                p.ws_ml[slot * 2 + 0] = failed ? -INFINITY : M;
                p.ws_ml[slot * 2 + 1] = failed ? -1.f : den;
            }
        }
    }
    __syncthreads();  // the merge scratch is read; the next unit may load into the rings
}

__device__ __forceinline__ uint8_t *aligned_smem(uint8_t *raw)
{
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                       ~static_cast<uintptr_t>(1023));
}

// ------------------------------------------------------------ the kernel
// Grid (partition, kv head, sequence); one partition = the whole context on
// the single-pass path.
template <typename T, int D, int BS, int G, bool TC>
__global__ void __launch_bounds__(DecodeCfg<T, D, BS, G, TC>::NW * 32)
pa_decode_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                 const __grid_constant__ CUtensorMap tmv)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = aligned_smem(smem_raw);
    const int part = blockIdx.x, kvh = blockIdx.y, seq = blockIdx.z;
    const int L = p.context_lens[seq];
    CtaWork w{seq, G, kvh, part * p.partition_size, 0, part, seq};
    if (L < 0 || L > p.max_context_len) {
        if (part == 0 && kvh == 0 && threadIdx.x == 0)
            report(p.status, PKV_DEV_BAD_CONTEXT_LEN);
        if (!p.split)
            write_invalid<D, G>(p, w);
        return;  // split path: the merge kernel sees the bad length itself
    }
    w.tok_end = min(w.tok0 + p.partition_size, L);
    if (w.tok0 >= w.tok_end) {
        if (!p.split && part == 0)
            write_invalid<D, G>(p, w);  // L == 0: zero output
        return;
    }
    init_rings<DecodeCfg<T, D, BS, G, TC>>(smem);
    int ring = 0;
    decode_cta<T, D, BS, G, TC, 1>(p, &tmk, &tmv, smem, w, ring);
    // split path: the merge grid, queued behind this one as a programmatic
    // dependent, may be scheduled once every CTA has stored its partials
    // (it waits for the whole grid before reading them)
    if (p.split)
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace pkv
