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

// Log-sum-exp merge of the partials, one warp per (sequence, head), four
// per CTA.  The valid slots are [0, ceil(S / P)) for a shared prefix of S
// tokens (shared-prefix path only) and [np_prefix, np_prefix + ceil((L - S) /
// P)).  Each lane owns D / 32 dims and keeps eight slots' loads in flight; the
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
    const int S = (!bad_len && p.seq_shared) ? p.seq_shared[seq] : 0;
    const int P = p.partition_size;
    const int na = S > 0 ? (S + P - 1) / P : 0;
    const int n = bad_len ? 0 : na + (L - S + P - 1) / P;
    auto slot_of = [&](int k) { return k < na ? k : p.np_prefix + (k - na); };
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

// Persistent over the planner's work list: CTA (x, kv head) takes items x,
// x + gridDim.x, ...  An item (seq, slot) with slot < np_prefix is prefix
// partition `slot` of the group that `seq` leads (all members' rows);
// otherwise it is tail partition slot - np_prefix of `seq` alone.  The list
// holds every prefix item before every tail item.
template <typename T, int D, int BS, int G, int NT>
__global__ void __launch_bounds__(DecodeCfg<T, D, BS, G, true>::NW * 32)
pa_shared_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                 const __grid_constant__ CUtensorMap tmv)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = aligned_smem(smem_raw);
    init_rings<DecodeCfg<T, D, BS, G, true>>(smem);
    int ring = 0;
    const int kvh = blockIdx.y;
    const int n = *p.num_items;
    const int P = p.partition_size;
    for (int i = blockIdx.x; i < n; i += gridDim.x) {
        const int2 it = p.items[i];
        const int seq = it.x, x = it.y;
        const int L = p.context_lens[seq];
        const int S = p.seq_shared[seq];
        CtaWork w;
        if (x < p.np_prefix) {
            const int t0 = x * P;
            w = CtaWork{seq, p.seq_members[seq] * G, kvh, t0, min(t0 + P, S), x, seq};
        } else {
            const int t0 = S + (x - p.np_prefix) * P;
            w = CtaWork{seq, G, kvh, t0, min(t0 + P, L), x, seq};
        }
        decode_cta<T, D, BS, G, true, NT>(p, &tmk, &tmv, smem, w, ring);
    }
}

}  // namespace pkv
