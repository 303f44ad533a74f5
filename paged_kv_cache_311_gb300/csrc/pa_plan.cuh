// pa_plan.cuh -- grouping of sequences that share leading blocks, for the
// shared-prefix decode path (see pa_shared.cuh).  Included by pkv_abi.cu only.
#pragma once

#include <stdint.h>

namespace pkv {

// One CTA: runs of consecutive sequences that start with the same block ids.
//   sp[s]         tokens sequence s shares with s - 1, rounded down to `align`
//                 (a multiple of the block size and of the tile), 0 if none
//   run_start[s]  first sequence of the run s belongs to
//   groups        chunks of at most max_members sequences of a run; the
//                 group's shared length is the smallest sp inside it
//   seq_shared[s] shared length of s's group (0: s reads all of its context)
//   members[s]    group size if s leads a group that shares tokens, else 0
__global__ void __launch_bounds__(1024)
pa_plan_kernel(const int32_t *__restrict__ block_tables, const int32_t *__restrict__ lens, int B,
               int MB, int bs, int max_len, int max_members, int align,
               int32_t *seq_shared, int32_t *members, int32_t *sp, int32_t *run_start)
{
    __shared__ int chunk_last[1024];
    const int tid = threadIdx.x, nthr = blockDim.x;
    for (int s = tid; s < B; s += nthr) {
        int v = 0;
        if (s > 0) {
            const int la = lens[s - 1], lb = lens[s];
            if (la > 0 && lb > 0 && la <= max_len && lb <= max_len) {
                const int n = min((la + bs - 1) / bs, (lb + bs - 1) / bs);
                const int32_t *ra = block_tables + (int64_t)(s - 1) * MB;
                const int32_t *rb = block_tables + (int64_t)s * MB;
                int c = 0;
                while (c < n && ra[c] == rb[c])
                    ++c;
                v = min(c * bs, min(la, lb));
                v = (v / align) * align;
            }
        }
        sp[s] = v;
    }
    __syncthreads();

    // run starts: inclusive max-scan of "sequence s starts a run" over chunks
    const int per = (B + nthr - 1) / nthr;
    const int lo = tid * per, hi = min(lo + per, B);
    int last = -1;
    for (int s = lo; s < hi; ++s)
        if (s == 0 || sp[s] == 0)
            last = s;
    chunk_last[tid] = last;
    __syncthreads();
    for (int off = 1; off < nthr; off <<= 1) {
        const int v = tid >= off ? max(chunk_last[tid], chunk_last[tid - off]) : chunk_last[tid];
        __syncthreads();
        chunk_last[tid] = v;
        __syncthreads();
    }
    int run = tid > 0 ? chunk_last[tid - 1] : -1;
    for (int s = lo; s < hi; ++s) {
        if (s == 0 || sp[s] == 0)
            run = s;
        run_start[s] = run;
    }
    __syncthreads();

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
        members[s] = S > 0 ? cnt : 0;
        for (int k = 0; k < cnt; ++k) {
            seq_shared[s + k] = S;
            if (k > 0)
                members[s + k] = 0;
        }
    }
}

}  // namespace pkv
