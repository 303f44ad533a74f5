// pa_merge.cuh -- the log-sum-exp merge of split-context partials
// (pa_merge_kernel).  The shared-prefix (cascade) kernel is in pa_cascade.cuh.
#pragma once

#include "pa_decode.cuh"

namespace pkv {

// Log-sum-exp merge of the partials, one warp per (sequence, head), four
// per CTA; the valid slots are the ceil(L / P) partitions of the context.
// Each lane owns D / 32 dims and keeps eight slots' loads in flight; the
// slots are added in their fixed order.
template <int D>
__global__ void __launch_bounds__(128) pa_merge_kernel(const __grid_constant__ DecodeParams p)
{
    constexpr int DPL = D / 32;
    constexpr int U = 8;
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
    auto slot_of = [](int k) { return k; };
    const float *ml = p.ws_ml + sh * p.num_partitions * 2;
    const float *accp = p.ws_acc + sh * p.num_partitions * D + lane * DPL;

    float M = -INFINITY;
    int invalid = 0;
    for (int k = lane; k < n; k += 32) {
        const int sl = slot_of(k);
        M = fmaxf(M, ml[2 * sl]);
        invalid |= ml[2 * sl + 1] < 0.f;
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
    for (int k0 = 0; k0 < n && !invalid; k0 += U) {
        float mm[U], ll[U], v[U][DPL];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            mm[u] = -INFINITY;
            ll[u] = 0.f;
            if (k0 + u < n) {
                const int sl = slot_of(k0 + u);
                mm[u] = ml[2 * sl];
                ll[u] = ml[2 * sl + 1];
                if constexpr (DPL == 4) {
                    const float4 t = *reinterpret_cast<const float4 *>(accp + (int64_t)sl * D);
                    v[u][0] = t.x; v[u][1] = t.y; v[u][2] = t.z; v[u][3] = t.w;
                } else {
                    const float2 t = *reinterpret_cast<const float2 *>(accp + (int64_t)sl * D);
                    v[u][0] = t.x; v[u][1] = t.y;
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
    const bool zero = invalid || bad_len || den == 0.f;
#pragma unroll
    for (int d = 0; d < DPL; ++d)
        store_out(p.out, p.out_dtype, sh * D + lane * DPL + d, zero ? 0.f : num[d] / den);
}

}  // namespace pkv
