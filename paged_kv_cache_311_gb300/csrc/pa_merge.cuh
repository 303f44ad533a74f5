// pa_merge.cuh -- the log-sum-exp merge of split-context partials: the
// half-warp routine merge_partials (pa_cascade_merge_kernel in
// pa_cascade.cuh runs it for the few partials of a shared-prefix plan) and
// pa_merge_kernel, one CTA per (sequence, head) after the split-context pass.
#pragma once

#include "pa_decode.cuh"

namespace pkv {

// Sixteen lanes (a half-warp; hl = lane within it) merge the partials of
// (sequence, head) `sh`, held in slots [0, n) of the split workspace (row
// stride `slots`), and write the output row:
//   out = sum_k 2^(m_k - M) acc_k / sum_k 2^(m_k - M) l_k,  M = max_k m_k.
// get_n() gives n: a count >= 0, kMergeZero to write a zero row, or
// kMergeSkip to leave the row untouched.  It is called after the first U
// slots' loads are issued -- they lie inside the row whatever n turns out to
// be, and slots >= n are ignored -- so a merge of up to U partials costs one
// round trip to L2 including the load behind n.  Later chunks of U rescale
// the running sums when they raise the maximum.  A partial with
// l < 0 marks a failed pass and zeroes the row.  Each lane owns D / 16
// dims; every lane reads the same (m, l) pairs, so no lane exchange is
// needed.  Loads bypass L1 (ld.global.cg).
constexpr int kMergeZero = -1, kMergeSkip = -2;

template <int D, int U, typename GetN>
__device__ __forceinline__ void merge_partials(const DecodeParams &p, int64_t sh, int slots, int hl,
                                               GetN get_n)
{
    constexpr int DPL = D / 16;   // dims per lane
    constexpr int V4 = DPL / 4;   // float4 pieces per lane
    const float2 *ml = reinterpret_cast<const float2 *>(p.ws_ml) + sh * slots;
    const float4 *acc = reinterpret_cast<const float4 *>(p.ws_acc + sh * slots * D + hl * DPL);

    float2 t[U];
    float4 a[U][V4];
    auto load_chunk = [&](int k0, int lim) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            t[u] = make_float2(-INFINITY, 0.f);
            if (k0 + u < lim) {
                t[u] = __ldcg(ml + k0 + u);
#pragma unroll
                for (int v = 0; v < V4; ++v)
                    a[u][v] = __ldcg(acc + (int64_t)(k0 + u) * (D / 4) + v);
            }
        }
    };
    load_chunk(0, slots < U ? slots : U);   // speculative: n is not known yet
    const int n = get_n();
    if (n == kMergeSkip)
        return;

    float M = -INFINITY, den = 0.f, num[DPL];
#pragma unroll
    for (int d = 0; d < DPL; ++d)
        num[d] = 0.f;
    bool invalid = n < 0;
    for (int k0 = 0; k0 < n && !invalid; k0 += U) {
        if (k0 > 0)
            load_chunk(k0, n);
        float Mc = M;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (k0 + u < n) {
                Mc = fmaxf(Mc, t[u].x);
                invalid |= t[u].y < 0.f;
            }
        }
        if (Mc == -INFINITY)
            continue;   // nothing attended so far
        const float s = exp2f(M - Mc);   // 0 while M is still -inf
        den *= s;
#pragma unroll
        for (int d = 0; d < DPL; ++d)
            num[d] *= s;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (k0 + u < n && t[u].x != -INFINITY) {
                const float f = exp2f(t[u].x - Mc);
                den += f * t[u].y;
#pragma unroll
                for (int v = 0; v < V4; ++v) {
                    num[4 * v + 0] += f * a[u][v].x;
                    num[4 * v + 1] += f * a[u][v].y;
                    num[4 * v + 2] += f * a[u][v].z;
                    num[4 * v + 3] += f * a[u][v].w;
                }
            }
        }
        M = Mc;
    }
    const bool zero = invalid || den == 0.f;
    const float inv = zero ? 0.f : 1.f / den;
#pragma unroll
    for (int v = 0; v < V4; ++v)
        store_out4(p.out, p.out_dtype, sh * D + hl * DPL + 4 * v,
                   make_float4(num[4 * v] * inv, num[4 * v + 1] * inv, num[4 * v + 2] * inv,
                               num[4 * v + 3] * inv));
}

// Merge after the split-context pass: one CTA of kSplitMergeWarps warps per
// (sequence, head), whose valid slots are the ceil(L / P) partitions of the
// context (64 at 32K tokens in 512-token partitions).  The partitions are
// dealt round-robin to the warps, and within a warp to SPI slot lanes (lane
// = sub-slot * (D / 4) + float4 piece), so that the loads of up to
// kSplitMergeWarps * SPI * kSplitMergeU partials leave together: a long
// context costs one round trip to L2, not one per chunk of slots.  Each lane
// keeps a running (max, sum, acc piece) over its slots; lanes of one piece
// combine by shuffles, then the warps in shared memory, each step the same
// log-sum-exp merge:
//   out = sum_k 2^(m_k - M) acc_k / sum_k 2^(m_k - M) l_k,  M = max_k m_k.
// A partial with l < 0 marks a failed pass and zeroes the row; so does a
// context length outside [0, max_context_len] (reported once per sequence).
constexpr int kSplitMergeWarps = 8, kSplitMergeU = 8;

template <int D>
__global__ void __launch_bounds__(kSplitMergeWarps * 32)
pa_merge_kernel(const __grid_constant__ DecodeParams p)
{
    constexpr int W = kSplitMergeWarps, U = kSplitMergeU;
    constexpr int PPR = D / 4;          // float4 pieces of a row
    static_assert(PPR <= 32 && 32 % PPR == 0, "a row's pieces fit one warp");
    constexpr int SPI = 32 / PPR;       // slots a warp reads side by side
    constexpr int ST = W * SPI;         // slot stride of one lane
    __shared__ float s_m[W], s_l[W];
    __shared__ int s_bad[W];
    __shared__ float4 s_acc[W][PPR];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int piece = lane % PPR, sub = lane / PPR;
    const int64_t sh = blockIdx.x;
    const int seq = (int)(sh / p.num_heads);
    const int slots = p.num_partitions;
    const int first = warp * SPI + sub;   // this lane's slots: first + j * ST
    const float2 *ml = reinterpret_cast<const float2 *>(p.ws_ml) + sh * slots;
    const float4 *acc = reinterpret_cast<const float4 *>(p.ws_acc + sh * slots * D) + piece;

    float2 t[U];
    float4 a[U];
    auto load_round = [&](int j0, int lim) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int k = first + (j0 + u) * ST;
            t[u] = make_float2(-INFINITY, 0.f);
            a[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (k < lim) {
                t[u] = __ldcg(ml + k);
                a[u] = __ldcg(acc + (int64_t)k * PPR);
            }
        }
    };
    // launched as a programmatic dependent of the partition pass: the
    // lengths (an input) may be read at once, the partials only after the
    // whole pass is done.  The first round's loads then leave before the
    // length they depend on is used: they lie inside the row's slots
    // whatever it turns out to be, and slots >= n are ignored below.
    const int L = p.context_lens[seq];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    load_round(0, slots);
    const bool bad_len = L < 0 || L > p.max_context_len;
    if (bad_len && threadIdx.x == 0 && sh % p.num_heads == 0)
        report(p.status, PKV_DEV_BAD_CONTEXT_LEN);   // the partition pass skipped it silently
    const int n = bad_len ? 0 : (L + p.partition_size - 1) / p.partition_size;

    float M = -INFINITY, den = 0.f;
    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
    bool invalid = bad_len;
    for (int j0 = 0; first + j0 * ST < n; j0 += U) {
        if (j0 > 0)
            load_round(j0, n);
        float Mc = M;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (first + (j0 + u) * ST < n) {
                Mc = fmaxf(Mc, t[u].x);
                invalid |= t[u].y < 0.f;
            }
        }
        if (Mc == -INFINITY)
            continue;   // nothing attended so far
        const float sc = exp2f(M - Mc);   // 0 while M is still -inf
        den *= sc;
        num.x *= sc;
        num.y *= sc;
        num.z *= sc;
        num.w *= sc;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (first + (j0 + u) * ST < n && t[u].x != -INFINITY) {
                const float f = exp2f(t[u].x - Mc);
                den += f * t[u].y;
                num.x += f * a[u].x;
                num.y += f * a[u].y;
                num.z += f * a[u].z;
                num.w += f * a[u].w;
            }
        }
        M = Mc;
    }
    // lanes holding the same piece for different sub-slots, then the warps
#pragma unroll
    for (int off = PPR; off < 32; off <<= 1) {
        const float Mo = __shfl_xor_sync(0xffffffffu, M, off);
        const float lo = __shfl_xor_sync(0xffffffffu, den, off);
        float4 no;
        no.x = __shfl_xor_sync(0xffffffffu, num.x, off);
        no.y = __shfl_xor_sync(0xffffffffu, num.y, off);
        no.z = __shfl_xor_sync(0xffffffffu, num.z, off);
        no.w = __shfl_xor_sync(0xffffffffu, num.w, off);
        invalid |= __shfl_xor_sync(0xffffffffu, (int)invalid, off) != 0;
        const float Mn = fmaxf(M, Mo);
        const float fa = M == -INFINITY ? 0.f : exp2f(M - Mn);
        const float fb = Mo == -INFINITY ? 0.f : exp2f(Mo - Mn);
        den = fa * den + fb * lo;
        num = make_float4(fa * num.x + fb * no.x, fa * num.y + fb * no.y, fa * num.z + fb * no.z,
                          fa * num.w + fb * no.w);
        M = Mn;
    }
    if (lane < PPR) {
        s_acc[warp][piece] = num;
        if (lane == 0) {
            s_m[warp] = M;
            s_l[warp] = den;
            s_bad[warp] = invalid;
        }
    }
    __syncthreads();
    if (threadIdx.x < PPR) {
        float Mt = -INFINITY;
        bool inv = false;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            Mt = fmaxf(Mt, s_m[w]);
            inv |= s_bad[w] != 0;
        }
        float dt = 0.f;
        float4 nt = make_float4(0.f, 0.f, 0.f, 0.f);
        if (Mt != -INFINITY) {
#pragma unroll
            for (int w = 0; w < W; ++w) {
                const float f = s_m[w] == -INFINITY ? 0.f : exp2f(s_m[w] - Mt);
                const float4 x = s_acc[w][threadIdx.x];
                dt += f * s_l[w];
                nt.x += f * x.x;
                nt.y += f * x.y;
                nt.z += f * x.z;
                nt.w += f * x.w;
            }
        }
        const bool zero = inv || dt == 0.f;
        const float inv_d = zero ? 0.f : 1.f / dt;
        store_out4(p.out, p.out_dtype, sh * D + 4 * threadIdx.x,
                   make_float4(nt.x * inv_d, nt.y * inv_d, nt.z * inv_d, nt.w * inv_d));
    }
}

}  // namespace pkv
