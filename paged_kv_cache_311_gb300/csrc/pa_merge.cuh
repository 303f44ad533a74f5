// pa_merge.cuh -- the log-sum-exp merge of split-context partials: the
// half-warp routine merge_partials (also called by the shared-prefix kernel
// in pa_cascade.cuh) and pa_merge_kernel, which runs it for every (sequence,
// head) after the split-context pass.
#pragma once

#include "pa_decode.cuh"

namespace pkv {

// Sixteen lanes (a half-warp; hl = lane within it) merge the n partials of
// (sequence, head) `sh`, held in slots [0, n) of the split workspace (row
// stride `slots`), and write the output row:
//   out = sum_k 2^(m_k - M) acc_k / sum_k 2^(m_k - M) l_k,  M = max_k m_k.
// A partial with l < 0 marks a failed pass and zeroes the row, as does
// `zero_row`.  Slots are read eight at a time, all loads of a chunk in
// flight together, with a running maximum (the sums are rescaled when a
// chunk raises it), so n <= 8 costs one round trip to L2.  Each lane owns
// D / 16 dims; every lane reads the same (m, l) pairs, so no lane exchange
// is needed.  Loads bypass L1 (ld.global.cg): partials written by other CTAs
// of the same launch are seen once their writers have released them.
template <int D>
__device__ __forceinline__ void merge_partials(const DecodeParams &p, int64_t sh, int n, int slots,
                                               bool zero_row, int hl)
{
    constexpr int DPL = D / 16;   // dims per lane
    constexpr int V4 = DPL / 4;   // float4 pieces per lane
    constexpr int U = 8;          // slots per chunk
    const float2 *ml = reinterpret_cast<const float2 *>(p.ws_ml) + sh * slots;
    const float4 *acc = reinterpret_cast<const float4 *>(p.ws_acc + sh * slots * D + hl * DPL);

    float M = -INFINITY, den = 0.f, num[DPL];
#pragma unroll
    for (int d = 0; d < DPL; ++d)
        num[d] = 0.f;
    bool invalid = zero_row;
    for (int k0 = 0; k0 < n && !invalid; k0 += U) {
        float2 t[U];
        float4 a[U][V4];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            t[u] = make_float2(-INFINITY, 0.f);
            if (k0 + u < n) {
                t[u] = __ldcg(ml + k0 + u);
#pragma unroll
                for (int v = 0; v < V4; ++v)
                    a[u][v] = __ldcg(acc + (int64_t)(k0 + u) * (D / 4) + v);
            }
        }
        float Mc = M;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            Mc = fmaxf(Mc, t[u].x);
            invalid |= t[u].y < 0.f;
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
            if (t[u].x != -INFINITY) {
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
    for (int d = 0; d < DPL; ++d)
        store_out(p.out, p.out_dtype, sh * D + hl * DPL + d, zero ? 0.f : num[d] * inv);
}

// Merge after the split-context pass: one half-warp per (sequence, head),
// eight per CTA; the valid slots are the ceil(L / P) partitions of the
// context.
template <int D>
__global__ void __launch_bounds__(128) pa_merge_kernel(const __grid_constant__ DecodeParams p)
{
    const int hw = threadIdx.x >> 4, hl = threadIdx.x & 15;
    const int64_t sh = (int64_t)blockIdx.x * 8 + hw;
    if (sh >= (int64_t)p.num_seqs * p.num_heads)
        return;
    const int seq = (int)(sh / p.num_heads);
    const int L = p.context_lens[seq];
    const bool bad_len = L < 0 || L > p.max_context_len;
    if (bad_len && hl == 0 && sh % p.num_heads == 0)
        report(p.status, PKV_DEV_BAD_CONTEXT_LEN);  // the partition pass skipped it silently
    const int P = p.partition_size;
    const int n = bad_len ? 0 : (L + P - 1) / P;
    merge_partials<D>(p, sh, n, p.num_partitions, bad_len, hl);
}

}  // namespace pkv
