// pkv_static_ws.cu -- paged decode attention for callers that cannot
// allocate device memory.
//
// Some callers have no way to obtain a workspace: plugins whose host engine
// owns every device allocation and hands them none, code running under an
// allocator that is already full or must not grow, and latency-critical
// loops that must not call cudaMalloc because it can synchronise the device.
// pkv_paged_attention_decode_static serves them.  When a context spans more
// than one partition it runs the split-context path (partition pass +
// log-sum-exp reduce) and keeps the partials in a fixed array that lives in
// this library (kStaticWsBytes per GPU, held from the first use of the
// library on that GPU until the process exits); a batch whose contexts fit
// one partition takes the single pass, which needs no workspace.  It never
// allocates.
//
// Host code cannot use the array's name as a device address, so each device
// gets the real address once, with that device current, from
// cudaGetSymbolAddress; the address is cached per device (a cudaDeviceReset
// invalidates it: the library must not be used across one).
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/pkv.h"
#include "pkv_host.cuh"

namespace pkv {
namespace {

constexpr size_t kStaticWsBytes = 32u << 20;   // 32 MiB per GPU
constexpr int kMaxDevices = 64;

// The shared workspace.  Every call on a device uses the same bytes; the
// partition pass writes every (max, sum, partial) slot that the reduce pass
// later reads, so nothing has to be cleared between calls.
static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

// Address of g_static_ws on device `dev` (which must be current).
int static_ws_address(int dev, void **out)
{
    if (dev < 0 || dev >= kMaxDevices)
        return PKV_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p)
            return PKV_ECUDA;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" {

size_t pkv_static_workspace_capacity(void) { return kStaticWsBytes; }

int pkv_paged_attention_decode_static(void *out, int out_dtype, const void *q,
                                      const void *k_cache, const void *v_cache, int kv_dtype,
                                      const int32_t *block_tables, int max_blocks_per_seq,
                                      const int32_t *context_lens, int num_seqs, int num_heads,
                                      int num_kv_heads, int head_dim, int block_size,
                                      int64_t num_blocks, int max_context_len, float scale,
                                      int partition_size, uint32_t *device_status, void *stream)
{
    if (partition_size < 0)
        return PKV_EINVAL;
    const int P = partition_size > 0 ? partition_size : PKV_DEFAULT_PARTITION;
    if (P % 32 || block_size <= 0 || P % block_size)
        return PKV_EINVAL;
    if (num_seqs < 0 || num_heads <= 0 || max_context_len < 0 || head_dim <= 0)
        return PKV_EINVAL;
    if (num_seqs == 0)
        return PKV_OK;
    // Sizes of the partials: (max, sum) pairs, then the fp32 accumulators,
    // laid out as the split path expects.
    const long long maxL = max_context_len > 0 ? max_context_len : 1;
    const long long np = (maxL + P - 1) / P;
    if (np == 1)   // one partition: the single pass, no workspace
        return pkv_paged_attention_decode(out, out_dtype, q, k_cache, v_cache, kv_dtype,
                                          block_tables, max_blocks_per_seq, context_lens, num_seqs,
                                          num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                                          max_context_len, scale, P, nullptr, 0, device_status,
                                          stream);
    // (sizes beyond 64 bits cannot fit either)
    uint64_t rows, acc;
    if (__builtin_mul_overflow((uint64_t)num_seqs, (uint64_t)num_heads, &rows) ||
        __builtin_mul_overflow(rows, (uint64_t)np, &rows) ||
        __builtin_mul_overflow(rows, (uint64_t)head_dim * sizeof(float), &acc) ||
        rows > kStaticWsBytes || acc > kStaticWsBytes)
        return PKV_EWORKSPACE;
    const size_t ml = (size_t)rows * 2 * sizeof(float);
    const size_t acc_off = (ml + 255) & ~size_t(255);
    const size_t need = acc_off + (size_t)acc;
    if (need > kStaticWsBytes)
        return PKV_EWORKSPACE;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return PKV_ECUDA;
    void *ws = nullptr;
    const int rc = static_ws_address(dev, &ws);
    if (rc != PKV_OK)
        return rc;
    // A partition size below the longest context forces the split path, the
    // only one that needs the workspace.
    return pkv_paged_attention_decode(out, out_dtype, q, k_cache, v_cache, kv_dtype, block_tables,
                                      max_blocks_per_seq, context_lens, num_seqs, num_heads,
                                      num_kv_heads, head_dim, block_size, num_blocks,
                                      max_context_len, scale, P, ws, kStaticWsBytes,
                                      device_status, stream);
}

}  // extern "C"
