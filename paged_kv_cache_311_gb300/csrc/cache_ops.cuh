// cache_ops.cuh -- the two cache-maintenance kernels: the scatter of new
// tokens into their slots and the copy-on-write block copy.
#pragma once

#include "pkv_device.cuh"

namespace pkv {

// reshape_and_cache (PagedAttention: Efficient LLM Serving with vLLM, "The
// PagedAttention Algorithm", Step 2): token t's rows key[t, h, :] and
// value[t, h, :] go to row slot % bs of physical block slot / bs, head h.
// One CTA per token; 16-byte vectors, so each (token, head) row is a run of
// D * e / 16 coalesced vector stores.
__global__ void __launch_bounds__(128)
reshape_and_cache_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                         uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                         const int64_t *__restrict__ slot_mapping, int num_kv_heads,
                         int row_vecs, int block_size, int64_t num_blocks, uint32_t *status)
{
    const int t = blockIdx.x;
    const int64_t slot = slot_mapping[t];
    if (slot < 0)
        return;  // padding token
    if (slot >= num_blocks * (int64_t)block_size) {
        if (threadIdx.x == 0)
            report(status, PKV_DEV_BAD_SLOT);
        return;
    }
    const int64_t b = slot / block_size;
    const int o = (int)(slot % block_size);
    const int total = num_kv_heads * row_vecs;
    const int64_t src0 = (int64_t)t * total;
    for (int v = threadIdx.x; v < total; v += blockDim.x) {
        const int h = v / row_vecs, c = v % row_vecs;
        const int64_t dst = ((b * num_kv_heads + h) * block_size + o) * row_vecs + c;
        k_cache[dst] = key[src0 + v];
        v_cache[dst] = value[src0 + v];
    }
}

constexpr int kCopyMaxLayers = 128;

struct CopyBlocksParams {
    uint4 *k[kCopyMaxLayers];
    uint4 *v[kCopyMaxLayers];
};

// copy_blocks ("Advanced Features", KV-Cache Sharing (Copy-on-Write)): grid
// (pair, layer, cache); each CTA copies one whole block of one cache.
__global__ void __launch_bounds__(256)
copy_blocks_kernel(const __grid_constant__ CopyBlocksParams ptrs, const int64_t *__restrict__ pairs,
                   int64_t block_vecs, int64_t num_blocks, uint32_t *status)
{
    const int pr = blockIdx.x, layer = blockIdx.y, which = blockIdx.z;
    const int64_t src = pairs[2 * pr], dst = pairs[2 * pr + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (threadIdx.x == 0 && layer == 0 && which == 0)
            report(status, PKV_DEV_BAD_BLOCK);
        return;
    }
    uint4 *base = which == 0 ? ptrs.k[layer] : ptrs.v[layer];
    const uint4 *s = base + src * block_vecs;
    uint4 *d = base + dst * block_vecs;
    for (int64_t i = threadIdx.x; i < block_vecs; i += blockDim.x)
        d[i] = s[i];
}

// swap_blocks (a preempted request's blocks go to CPU memory when the GPU is
// full and come back when it resumes: PagedAttention: Efficient LLM Serving
// with vLLM, "vLLM: The Serving Engine"): grid (pair, layer, K/V), one CTA
// moves one block between the GPU pool and a pinned, device-mapped host pool
// over the host link.  One launch moves any number of blocks, so small blocks
// cost no transfer each.  Each thread keeps four 16-byte loads in flight.
constexpr int kSwapMaxLayers = 64;

struct SwapBlocksParams {
    uint4 *gpu_k[kSwapMaxLayers];
    uint4 *gpu_v[kSwapMaxLayers];
    uint4 *host_k[kSwapMaxLayers];
    uint4 *host_v[kSwapMaxLayers];
};

__global__ void __launch_bounds__(256)
swap_blocks_kernel(const __grid_constant__ SwapBlocksParams ptrs, const int64_t *__restrict__ pairs,
                   int64_t block_vecs, int64_t gpu_blocks, int64_t host_blocks, int to_host,
                   uint32_t *status)
{
    const int pr = blockIdx.x, layer = blockIdx.y, which = blockIdx.z;
    const int64_t g = pairs[2 * pr], h = pairs[2 * pr + 1];
    if (g < 0 || g >= gpu_blocks || h < 0 || h >= host_blocks) {
        if (threadIdx.x == 0 && layer == 0 && which == 0)
            report(status, PKV_DEV_BAD_BLOCK);
        return;
    }
    uint4 *gb = (which == 0 ? ptrs.gpu_k[layer] : ptrs.gpu_v[layer]) + g * block_vecs;
    uint4 *hb = (which == 0 ? ptrs.host_k[layer] : ptrs.host_v[layer]) + h * block_vecs;
    const uint4 *src = to_host ? gb : hb;
    uint4 *dst = to_host ? hb : gb;
    constexpr int U = 4;
    for (int64_t i0 = threadIdx.x; i0 < block_vecs; i0 += U * blockDim.x) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = i0 + (int64_t)u * blockDim.x;
            if (i < block_vecs)
                v[u] = src[i];
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = i0 + (int64_t)u * blockDim.x;
            if (i < block_vecs)
                dst[i] = v[u];
        }
    }
}

// Test hook of the bounded waits: one CTA waits on an mbarrier whose phase
// nothing completes (no thread arrives, no copy is issued), with the same
// bounded wait the decode kernels use, so the wait must give up; then the
// drain that follows a timeout in those kernels runs on the same phase and
// gives up too.  Expected result: PKV_DEV_TIMEOUT | PKV_DEV_DRAIN_TIMEOUT in
// *status, and a kernel that returns.
__global__ void __launch_bounds__(32)
bounded_wait_test_kernel(uint64_t limit_ns, uint64_t max_polls, uint32_t *status)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (!mbar_wait_bounded(&bar, 0, limit_ns, max_polls)) {
        if (threadIdx.x == 0)
            report(status, PKV_DEV_TIMEOUT);
        drain_wait(&bar, 0, threadIdx.x == 0 ? status : nullptr, limit_ns, max_polls);
    }
}

}  // namespace pkv
