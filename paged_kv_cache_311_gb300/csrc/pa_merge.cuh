// pa_merge.cuh -- the log-sum-exp merge of split-context partials: the warp
// routine merge_partials (also called by the shared-prefix kernel in
// pa_cascade.cuh) and pa_merge_kernel, which runs it for every (sequence,
// head) after the split-context pass.
#pragma once

#include "pa_decode.cuh"

namespace pkv {

// One warp merges the n partials of (sequence, head) `sh`, held in slots
// [0, n) of the split workspace (row stride `slots`), and writes the output
// row: out = sum_k 2^(m_k - M) acc_k / sum_k 2^(m_k - M) l_k with M the
// largest m_k.  A partial with l < 0 marks a failed pass and zeroes the row,
// as does `zero_row`.  Each lane owns D / 32 dims and keeps eight slots'
// loads in flight; the slots are added in their fixed order.  Loads go
// through L2 only (ld.global.cg), so partials written by other CTAs of the
// same launch are seen once their writers have fenced.
template <int D>
__device__ __forceinline__ void merge_partials(const DecodeParams &p, int64_t sh, int n, int slots,
                                               bool zero_row, int lane)
{
    constexpr int DPL = D / 32;
    constexpr int U = 8;
    const float *ml = p.ws_ml + sh * slots * 2;
    const float *accp = p.ws_acc + sh * slots * D + lane * DPL;

    float M = -INFINITY;
    int invalid = 0;
    for (int k = lane; k < n; k += 32) {
        const float2 t = __ldcg(reinterpret_cast<const float2 *>(ml) + k);
        M = fmaxf(M, t.x);
        invalid |= t.y < 0.f;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    invalid = __any_sync(0xffffffffu, invalid);

    float num[DPL];
#pragma unroll
    for (int d = 0; d < DPL; ++d)
        num[d] = 0.f;
    float den = 0.f;
    for (int k0 = 0; k0 < n && !invalid && !zero_row; k0 += U) {
        float mm[U], ll[U], v[U][DPL];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            mm[u] = -INFINITY;
            ll[u] = 0.f;
            if (k0 + u < n) {
                const int sl = k0 + u;
                const float2 t = __ldcg(reinterpret_cast<const float2 *>(ml) + sl);
                mm[u] = t.x;
                ll[u] = t.y;
                if constexpr (DPL == 4) {
                    const float4 a = __ldcg(reinterpret_cast<const float4 *>(accp + (int64_t)sl * D));
                    v[u][0] = a.x; v[u][1] = a.y; v[u][2] = a.z; v[u][3] = a.w;
                } else {
                    const float2 a = __ldcg(reinterpret_cast<const float2 *>(accp + (int64_t)sl * D));
                    v[u][0] = a.x; v[u][1] = a.y;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (mm[u] != -INFINITY) {
                const float f = exp2f(mm[u] - M);
                den += f * ll[u];
#pragma unroll
                for (int d = 0; d < DPL; ++d)
                    num[d] += f * v[u][d];
            }
        }
    }
    const bool zero = invalid || zero_row || den == 0.f;
#pragma unroll
    for (int d = 0; d < DPL; ++d)
        store_out(p.out, p.out_dtype, sh * D + lane * DPL + d, zero ? 0.f : num[d] / den);
}

// Merge after the split-context pass: one warp per (sequence, head), four
// per CTA; the valid slots are the ceil(L / P) partitions of the context.
template <int D>
__global__ void __launch_bounds__(128) pa_merge_kernel(const __grid_constant__ DecodeParams p)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t sh = (int64_t)blockIdx.x * 4 + warp;
    if (sh >= (int64_t)p.num_seqs * p.num_heads)
        return;
    const int seq = (int)(sh / p.num_heads);
    const int L = p.context_lens[seq];
    const bool bad_len = L < 0 || L > p.max_context_len;
    if (bad_len && lane == 0 && sh % p.num_heads == 0)
        report(p.status, PKV_DEV_BAD_CONTEXT_LEN);  // the partition pass skipped it silently
    const int P = p.partition_size;
    const int n = bad_len ? 0 : (L + P - 1) / P;
    merge_partials<D>(p, sh, n, p.num_partitions, bad_len, lane);
}

}  // namespace pkv
