// pa_shared.cuh -- the log-sum-exp merge of split-context partials, and the
// shared-prefix decode path.
//
// Shared prefixes (PagedAttention: Efficient LLM Serving with vLLM,
// "Advanced Features", KV-Cache Sharing): sequences forked from one prompt
// (parallel sampling, beam search, a common system prompt) point their block
// tables at the same physical blocks for the shared part.  A per-sequence
// kernel reads those blocks once per sequence.  Here pa_plan_kernel finds
// runs of consecutive sequences whose tables start with the same block ids,
// and pa_shared_kernel reads every shared block once for the whole group:
// one CTA per (prefix partition, kv head, group) computes up to 24 query rows
// (all heads of all members) from the same tiles, while each member's own
// tail goes through a per-sequence CTA.  Both write partials that
// pa_merge_kernel combines per (sequence, head).  pa_plan_kernel (pa_plan.cuh)
// finds the groups.
#pragma once

#include "pa_decode.cuh"

namespace pkv {

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


// Grid (np_prefix + tail partitions, kv head, sequence).  x < np_prefix:
// prefix partition x of the group that sequence z leads (all members' rows);
// otherwise tail partition x - np_prefix of sequence z alone.
template <typename T, int D, int BS, int G, int NT>
__global__ void __launch_bounds__(DecodeCfg<T, D, BS, G, true>::NW * 32)
pa_shared_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                 const __grid_constant__ CUtensorMap tmv)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = aligned_smem(smem_raw);
    const int x = blockIdx.x, kvh = blockIdx.y, seq = blockIdx.z;
    const int L = p.context_lens[seq];
    if (L < 0 || L > p.max_context_len)
        return;  // the merge kernel zeroes the rows and reports the length
    const int S = p.seq_shared[seq];
    const int P = p.partition_size;
    CtaWork w;
    if (x < p.np_prefix) {
        const int m = p.seq_members[seq];
        const int t0 = x * P;
        if (m == 0 || t0 >= S)
            return;
        w = CtaWork{seq, m * G, kvh, t0, min(t0 + P, S), x, seq};
    } else {
        const int t0 = S + (x - p.np_prefix) * P;
        if (t0 >= L)
            return;
        w = CtaWork{seq, G, kvh, t0, min(t0 + P, L), x, seq};
    }
    decode_cta<T, D, BS, G, true, NT>(p, &tmk, &tmv, smem, w);
}

}  // namespace pkv
