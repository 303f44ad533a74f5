// pa_merge.cuh -- the log-sum-exp merge of split-context partials: the
// half-warp routine merge_partials (also used by pa_cascade_merge_kernel in
// pa_cascade.cuh) and pa_merge_kernel, which runs it for every (sequence,
// head) after the split-context pass.
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

// Merge after the split-context pass: one half-warp per (sequence, head),
// eight per CTA; the valid slots are the ceil(L / P) partitions of the
// context (up to 64 and more for long contexts: chunks of eight slots).
template <int D>
__global__ void __launch_bounds__(128) pa_merge_kernel(const __grid_constant__ DecodeParams p)
{
    const int hw = threadIdx.x >> 4, hl = threadIdx.x & 15;
    const int64_t sh = (int64_t)blockIdx.x * 8 + hw;
    if (sh >= (int64_t)p.num_seqs * p.num_heads)
        return;
    const int seq = (int)(sh / p.num_heads);
    merge_partials<D, 8>(p, sh, p.num_partitions, hl, [&]() {
        const int L = p.context_lens[seq];
        if (L < 0 || L > p.max_context_len) {
            if (hl == 0 && sh % p.num_heads == 0)
                report(p.status, PKV_DEV_BAD_CONTEXT_LEN);  // the partition pass skipped it silently
            return kMergeZero;
        }
        return (L + p.partition_size - 1) / p.partition_size;
    });
}

}  // namespace pkv
