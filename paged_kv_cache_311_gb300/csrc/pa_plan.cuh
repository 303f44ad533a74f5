// pa_plan.cuh -- planning for the shared-prefix decode path (pa_shared.cuh):
// which consecutive sequences share leading physical blocks, how they are
// grouped, and the list of work items.  Included by pkv_abi.cu only.
#pragma once

#include <stdint.h>

namespace pkv {

// Exclusive prefix sum of one int per sequence over a single CTA: thread t
// owns the chunk [lo, hi); `scan` is 1024 ints of shared memory.  Returns the
// total; out[s] receives the offset of sequence s.
template <typename F>
__device__ int cta_exclusive_sum(int B, int lo, int hi, int *scan, int32_t *out, F count)
{
    const int tid = threadIdx.x, nthr = blockDim.x;
    int local = 0;
    for (int s = lo; s < hi; ++s)
        local += count(s);
    scan[tid] = local;
    __syncthreads();
    for (int off = 1; off < nthr; off <<= 1) {
        const int v = tid >= off ? scan[tid] + scan[tid - off] : scan[tid];
        __syncthreads();
        scan[tid] = v;
        __syncthreads();
    }
    int run = tid > 0 ? scan[tid - 1] : 0;
    const int total = scan[nthr - 1];
    for (int s = lo; s < hi; ++s) {
        out[s] = run;
        run += count(s);
    }
    __syncthreads();
    return total;
}

// One CTA of 1024 threads.
//   sp[s]         tokens sequence s shares with s - 1 (equal leading block
//                 ids, within both contexts), rounded down to `align` (a
//                 multiple of the block size and of the tile); 0 if none
//   run_start[s]  first sequence of the run of sharing sequences s is in
//   groups        chunks of at most max_members sequences of a run; a group
//                 shares the smallest sp inside it
//   seq_shared[s] shared length of s's group (0: s reads its whole context)
//   members[s]    group size if s leads a group that shares tokens, else 0
//   items         (sequence, slot): prefix partitions of every group (slots
//                 < np_prefix), then the tail partitions of every sequence
__global__ void __launch_bounds__(1024)
pa_plan_kernel(const int32_t *__restrict__ block_tables, const int32_t *__restrict__ lens, int B,
               int MB, int bs, int max_len, int max_members, int align, int P, int np_prefix,
               int32_t *seq_shared, int32_t *members, int32_t *sp, int32_t *run_start,
               int2 *items, int *num_items)
{
    __shared__ int scan[1024];
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;

    // ---- 1: shared tokens with the previous sequence; one warp compares 32
    // table entries at a time, for four sequences at once
    constexpr int U = 4;
    for (int s0 = warp; s0 < B; s0 += nwarps * U) {
        int n[U], la[U], lb[U], first[U];
        bool done[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int s = s0 + u * nwarps;
            la[u] = (s > 0 && s < B) ? lens[s - 1] : 0;
            lb[u] = (s > 0 && s < B) ? lens[s] : 0;
            const bool ok = la[u] > 0 && lb[u] > 0 && la[u] <= max_len && lb[u] <= max_len;
            n[u] = ok ? min((la[u] + bs - 1) / bs, (lb[u] + bs - 1) / bs) : 0;
            first[u] = n[u];
            done[u] = n[u] == 0;
        }
        for (int c0 = 0;; c0 += 32) {
            bool more = false;
            int a[U], b[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int s = s0 + u * nwarps, j = c0 + lane;
                const bool live = !done[u] && j < n[u];
                a[u] = live ? block_tables[(int64_t)(s - 1) * MB + j] : 0;
                b[u] = live ? block_tables[(int64_t)s * MB + j] : 0;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (done[u])
                    continue;
                const unsigned diff = __ballot_sync(0xffffffffu, c0 + lane < n[u] && a[u] != b[u]);
                if (diff) {
                    first[u] = c0 + __ffs(diff) - 1;
                    done[u] = true;
                } else if (c0 + 32 >= n[u]) {
                    done[u] = true;
                } else {
                    more = true;
                }
            }
            if (!more)
                break;
        }
        if (lane == 0) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int s = s0 + u * nwarps;
                if (s >= B)
                    continue;
                int v = n[u] ? min(first[u] * bs, min(la[u], lb[u])) : 0;
                sp[s] = (v / align) * align;
            }
        }
    }
    __syncthreads();

    // ---- 2: run starts: inclusive max-scan of "s starts a run" over chunks
    const int per = (B + nthr - 1) / nthr;
    const int lo = min(tid * per, B), hi = min(lo + per, B);
    int last = -1;
    for (int s = lo; s < hi; ++s)
        if (s == 0 || sp[s] == 0)
            last = s;
    scan[tid] = last;
    __syncthreads();
    for (int off = 1; off < nthr; off <<= 1) {
        const int v = tid >= off ? max(scan[tid], scan[tid - off]) : scan[tid];
        __syncthreads();
        scan[tid] = v;
        __syncthreads();
    }
    int run = tid > 0 ? scan[tid - 1] : -1;
    for (int s = lo; s < hi; ++s) {
        if (s == 0 || sp[s] == 0)
            run = s;
        run_start[s] = run;
    }
    __syncthreads();

    // ---- 3: groups of at most max_members sequences within a run
    for (int s = tid; s < B; s += nthr) {
        const int rs = run_start[s];
        if ((s - rs) % max_members != 0)
            continue;  // not a group leader
        int cnt = 1, S = 0x7fffffff;
        while (cnt < max_members && s + cnt < B && run_start[s + cnt] == rs) {
            S = min(S, sp[s + cnt]);
            ++cnt;
        }
        if (cnt < 2)
            S = 0;
        for (int k = 0; k < cnt; ++k) {
            seq_shared[s + k] = S;
            members[s + k] = (k == 0 && S > 0) ? cnt : 0;
        }
    }
    __syncthreads();

    // ---- 4: work items, prefix partitions first (they are the heavy ones)
    auto n_pre = [&](int s) { return members[s] > 0 ? (seq_shared[s] + P - 1) / P : 0; };
    auto n_tail = [&](int s) {
        const int L = lens[s];
        return (L < 0 || L > max_len) ? 0 : (L - seq_shared[s] + P - 1) / P;
    };
    const int total_pre = cta_exclusive_sum(B, lo, hi, scan, sp, n_pre);
    for (int s = lo; s < hi; ++s)
        for (int x = 0, k = n_pre(s); x < k; ++x)
            items[sp[s] + x] = make_int2(s, x);
    __syncthreads();
    const int total_tail = cta_exclusive_sum(B, lo, hi, scan, run_start, n_tail);
    for (int s = lo; s < hi; ++s)
        for (int x = 0, k = n_tail(s); x < k; ++x)
            items[total_pre + run_start[s] + x] = make_int2(s, np_prefix + x);
    if (tid == 0)
        *num_items = total_pre + total_tail;
}

}  // namespace pkv
