// pkv_abi.cu -- the extern "C" boundary of libpkv.so (declared in
// include/pkv.h): host-side validation, path selection and kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <mutex>

#include "../../include/pkv.h"
#include "cache_ops.cuh"
#include "cascade_plan.h"
#include "pkv_host.cuh"

namespace pkv {

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

int current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return -1;
    return dev;
}

int sm_count(int dev)
{
    static std::atomic<int> cache[64];
    if (dev < 0 || dev >= 64)
        return 152;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0)
        return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
        v = 152;
    cache[dev].store(v, std::memory_order_relaxed);
    return v;
}

thread_local int g_last_decode_launches = 0;
thread_local int g_last_decode_engine = 0;
std::atomic<int> g_engine_override{0};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_bytes(int dtype) { return dtype == PKV_F32 ? 4 : 2; }
bool valid_dtype(int dtype) { return dtype == PKV_F32 || dtype == PKV_F16 || dtype == PKV_BF16; }

constexpr int kTableCap = 1024;   // block-table entries one decode CTA stages
constexpr int kTileAlign = 32;    // partition sizes are multiples of this

struct SplitLayout {
    size_t ml_bytes;
    size_t acc_off;
    size_t total;
};

// False when the sizes do not fit in 64 bits (no real call comes near).
bool split_layout(uint64_t seqs, uint64_t heads, uint64_t np, uint64_t head_dim, SplitLayout *s)
{
    uint64_t rows, ml, acc;
    if (__builtin_mul_overflow(seqs, heads, &rows) || __builtin_mul_overflow(rows, np, &rows) ||
        __builtin_mul_overflow(rows, (uint64_t)(2 * sizeof(float)), &ml) ||
        __builtin_mul_overflow(rows, head_dim * sizeof(float), &acc) || ml > UINT64_MAX - 256 ||
        ((ml + 255) & ~uint64_t(255)) > UINT64_MAX - acc)
        return false;
    s->ml_bytes = (size_t)ml;
    s->acc_off = (size_t)((ml + 255) & ~uint64_t(255));
    s->total = s->acc_off + (size_t)acc;
    return true;
}

}  // namespace

int encode_kv_map(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int eb,
                  int head_dim, int block_size, int num_kv_heads, int64_t num_blocks, int box_rows,
                  int box_chunks)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return PKV_ECUDA;
    const cuuint64_t row = (cuuint64_t)head_dim * eb;
    const cuuint64_t dims[5] = {(cuuint64_t)(128 / eb), (cuuint64_t)block_size, row / 128,
                                (cuuint64_t)num_kv_heads, (cuuint64_t)num_blocks};
    const cuuint64_t strides[4] = {row, 128, row * block_size, row * block_size * num_kv_heads};
    const cuuint32_t box[5] = {(cuuint32_t)(128 / eb), (cuuint32_t)box_rows,
                               (cuuint32_t)(box_chunks > 0 ? box_chunks : row / 128), 1, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(map, dtype, 5, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PKV_OK : PKV_ECUDA;
}

int ensure_smem_attr(const void *func, int bytes, unsigned long long *done_mask)
{
    const int dev = current_device();
    if (dev < 0)
        return PKV_ECUDA;
    const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit && (__atomic_load_n(done_mask, __ATOMIC_ACQUIRE) & bit))
        return PKV_OK;
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
        cudaSuccess)
        return PKV_ECUDA;
    // every library kernel asks for the largest shared-memory carveout, so
    // that consecutive launches of them never wait for an L1 / shared
    // memory reconfiguration of the SMs
    if (cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess)
        return PKV_ECUDA;
    if (bit)
        __atomic_fetch_or(done_mask, bit, __ATOMIC_RELEASE);
    return PKV_OK;
}

}  // namespace pkv

using namespace pkv;

extern "C" {

const char *pkv_status_string(int status)
{
    switch (status) {
    case PKV_OK: return "ok";
    case PKV_EINVAL: return "invalid argument (pointer, size, shape or alignment)";
    case PKV_EUNSUPPORTED: return "unsupported configuration (head_dim, block_size, group or dtype)";
    case PKV_ECUDA: return "CUDA runtime or driver call failed";
    case PKV_EWORKSPACE: return "workspace missing or too small";
    case PKV_EHOSTMEM: return "host memory allocation failed";
    default: return "unknown status";
    }
}

int pkv_last_decode_launches(void) { return g_last_decode_launches; }

int pkv_last_decode_engine(void) { return g_last_decode_engine; }

int pkv_decode_set_engine(int engine)
{
    if (engine < kEngineAuto || engine > kEngineTcgen05)
        return PKV_EINVAL;
    g_engine_override.store(engine, std::memory_order_relaxed);
    pkv::set_shared_plan_engine(engine);   // the automatic shared-prefix plan follows the kernel
    return PKV_OK;
}

size_t pkv_paged_attention_workspace_bytes(int num_seqs, int num_heads, int max_context_len,
                                           int head_dim, int partition_size)
{
    if (num_seqs <= 0 || num_heads <= 0 || max_context_len <= 0 || head_dim <= 0 ||
        partition_size < 0)
        return 0;
    const int P = partition_size > 0 ? partition_size : PKV_DEFAULT_PARTITION;
    const long long np = ((long long)max_context_len + P - 1) / P;
    if (np <= 1)
        return 0;
    SplitLayout s;
    return split_layout((uint64_t)num_seqs, (uint64_t)num_heads, (uint64_t)np, (uint64_t)head_dim, &s)
               ? s.total : 0;
}

int pkv_paged_attention_decode(void *out, int out_dtype, const void *q, const void *k_cache,
                               const void *v_cache, int kv_dtype, const int32_t *block_tables,
                               int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                               int num_heads, int num_kv_heads, int head_dim, int block_size,
                               int64_t num_blocks, int max_context_len, float scale,
                               int partition_size, void *workspace, size_t workspace_bytes,
                               uint32_t *device_status, void *stream)
{
    g_last_decode_launches = 0;
    g_last_decode_engine = 0;
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0)
        return PKV_EINVAL;
    if (!valid_dtype(out_dtype) || !valid_dtype(kv_dtype))
        return PKV_EINVAL;
    if (num_blocks <= 0 || num_blocks > INT32_MAX || max_blocks_per_seq <= 0 || block_size <= 0 ||
        max_context_len < 0 || partition_size < 0 || !std::isfinite(scale))
        return PKV_EINVAL;
    if ((long long)max_context_len > (long long)max_blocks_per_seq * block_size)
        return PKV_EINVAL;
    if (num_seqs == 0)
        return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return PKV_EINVAL;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return PKV_EINVAL;
    const int group = num_heads / num_kv_heads;
    if (head_dim != 64 && head_dim != 128)
        return PKV_EUNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32)
        return PKV_EUNSUPPORTED;
    if (group != 1 && group != 2 && group != 4 && group != 8)
        return PKV_EUNSUPPORTED;
    if (num_kv_heads > 65535 || num_seqs > 65535)
        return PKV_EUNSUPPORTED;  // grid.y / grid.z limits

    const int dev = current_device();
    if (dev < 0)
        return PKV_ECUDA;
    const int maxL = max_context_len > 0 ? max_context_len : 1;

    // Path choice: one CTA per (sequence, kv head) when that fills the GPU
    // and the whole block-table row fits in shared memory; otherwise split
    // the context into partitions and merge them with the reduce kernel.
    int P;
    if (partition_size > 0) {
        if (partition_size % kTileAlign || partition_size % block_size)
            return PKV_EINVAL;
        P = partition_size;
    } else {
        const long long ctas = (long long)num_seqs * num_kv_heads;
        const bool fits = ((long long)maxL + block_size - 1) / block_size <= kTableCap;
        const bool fills = ctas >= 4LL * sm_count(dev);
        P = (fits && fills) ? maxL : PKV_DEFAULT_PARTITION;
    }
    long long np = (maxL + (long long)P - 1) / P;
    if (np < 1)
        np = 1;
    if (np > 65535)
        return PKV_EUNSUPPORTED;
    // every CTA stages its partition's block-table slice in shared memory
    const long long part_tokens = np == 1 ? maxL : P;
    if ((part_tokens + block_size - 1) / block_size > kTableCap)
        return PKV_EUNSUPPORTED;

    DecodeLaunch a;
    DecodeParams &p = a.p;
    p.out = out;
    p.q = q;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.ws_ml = nullptr;
    p.ws_acc = nullptr;
    p.status = device_status;
    p.num_blocks = num_blocks;
    p.num_seqs = num_seqs;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.max_context_len = max_context_len;
    p.partition_size = np == 1 ? maxL : P;
    p.num_partitions = (int)np;
    p.out_dtype = out_dtype;
    p.split = np > 1;
    p.qscale = scale * 1.4426950408889634f;  // log2(e): softmax via exp2
    if (p.split) {
        SplitLayout s;
        if (!split_layout((uint64_t)num_seqs, (uint64_t)num_heads, (uint64_t)np, (uint64_t)head_dim, &s))
            return PKV_EUNSUPPORTED;
        if (!workspace || workspace_bytes < s.total || !aligned16(workspace))
            return PKV_EWORKSPACE;
        p.ws_ml = static_cast<float *>(workspace);
        p.ws_acc = reinterpret_cast<float *>(static_cast<char *>(workspace) + s.acc_off);
    }
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.head_dim = head_dim;
    a.block_size = block_size;
    a.group = group;
    a.engine = g_engine_override.load(std::memory_order_relaxed);
    a.shared = false;
    a.plan = nullptr;
    a.num_lists = 0;
    a.p.num_items = 0;
    a.stream = static_cast<cudaStream_t>(stream);
    int engine_used = 0;
    a.engine_used = &engine_used;

    int rc;
    switch (kv_dtype) {
    case PKV_F32: rc = launch_decode_f32(a); break;
    case PKV_F16: rc = launch_decode_f16(a); break;
    default: rc = launch_decode_bf16(a); break;
    }
    if (rc == PKV_OK) {
        g_last_decode_launches = p.split ? 2 : 1;
        g_last_decode_engine = engine_used;
    }
    return rc;
}

int pkv_paged_attention_decode_shared(void *out, int out_dtype, const void *q, const void *k_cache,
                                      const void *v_cache, int kv_dtype,
                                      const int32_t *block_tables, int max_blocks_per_seq,
                                      const int32_t *context_lens, int num_seqs, int num_heads,
                                      int num_kv_heads, int head_dim, int block_size,
                                      int64_t num_blocks, int max_context_len, float scale,
                                      const int32_t *plan, int num_lists, int num_items, int slots,
                                      void *workspace, size_t workspace_bytes,
                                      uint32_t *device_status, void *stream)
{
    g_last_decode_launches = 0;
    g_last_decode_engine = 0;
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0)
        return PKV_EINVAL;
    if (!valid_dtype(out_dtype) || !valid_dtype(kv_dtype))
        return PKV_EINVAL;
    if (num_blocks <= 0 || num_blocks > INT32_MAX || max_blocks_per_seq <= 0 || block_size <= 0 ||
        max_context_len < 0 || !std::isfinite(scale))
        return PKV_EINVAL;
    if ((long long)max_context_len > (long long)max_blocks_per_seq * block_size)
        return PKV_EINVAL;
    if (num_seqs == 0)
        return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !plan)
        return PKV_EINVAL;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(plan) & 3u))
        return PKV_EINVAL;
    if (num_lists <= 0 || num_lists > 65535 || num_items < num_lists || slots <= 0)
        return PKV_EINVAL;
    const int group = num_heads / num_kv_heads;
    if (kv_dtype == PKV_F32 || (head_dim != 64 && head_dim != 128) ||
        (block_size != 8 && block_size != 16 && block_size != 32) ||
        (group != 1 && group != 2 && group != 4 && group != 8))
        return PKV_EUNSUPPORTED;
    if (num_kv_heads > 65535)
        return PKV_EUNSUPPORTED;
    SplitLayout lay;
    if (!split_layout((uint64_t)num_seqs, (uint64_t)num_heads, (uint64_t)slots, (uint64_t)head_dim, &lay))
        return PKV_EUNSUPPORTED;
    if (!workspace || workspace_bytes < lay.total || !aligned16(workspace))
        return PKV_EWORKSPACE;

    DecodeLaunch a;
    DecodeParams &p = a.p;
    p.out = out;
    p.q = q;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.ws_ml = static_cast<float *>(workspace);
    p.ws_acc = reinterpret_cast<float *>(static_cast<char *>(workspace) + lay.acc_off);
    p.status = device_status;
    p.num_blocks = num_blocks;
    p.num_seqs = num_seqs;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.max_context_len = max_context_len;
    p.partition_size = 0;
    p.num_partitions = slots;
    p.out_dtype = out_dtype;
    p.split = 1;
    p.qscale = scale * 1.4426950408889634f;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.head_dim = head_dim;
    a.block_size = block_size;
    a.group = group;
    a.engine = g_engine_override.load(std::memory_order_relaxed);
    a.shared = true;
    a.plan = plan;
    a.num_lists = num_lists;
    p.num_items = num_items;
    a.stream = static_cast<cudaStream_t>(stream);
    int engine_used = 0;
    a.engine_used = &engine_used;
    const int rc = kv_dtype == PKV_F16 ? launch_decode_f16(a) : launch_decode_bf16(a);
    if (rc == PKV_OK) {
        g_last_decode_launches = 2;
        g_last_decode_engine = engine_used;
    }
    return rc;
}

int pkv_reshape_and_cache(const void *key, const void *value, void *k_cache, void *v_cache,
                          int dtype, const int64_t *slot_mapping, int num_tokens,
                          int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                          uint32_t *device_status, void *stream)
{
    if (!valid_dtype(dtype) || num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || num_blocks <= 0)
        return PKV_EINVAL;
    if ((int64_t)head_dim * elem_bytes(dtype) > INT32_MAX)
        return PKV_EINVAL;
    const int row_bytes = head_dim * elem_bytes(dtype);
    if (row_bytes % 16)
        return PKV_EINVAL;
    if (num_tokens == 0)
        return PKV_OK;
    if (!key || !value || !k_cache || !v_cache || !slot_mapping)
        return PKV_EINVAL;
    if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
        return PKV_EINVAL;
    static unsigned long long scatter_attr = 0;
    if (ensure_smem_attr(reinterpret_cast<const void *>(reshape_and_cache_kernel), 0, &scatter_attr))
        return PKV_ECUDA;
    reshape_and_cache_kernel<<<num_tokens, 128, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4 *>(key), static_cast<const uint4 *>(value),
        static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), slot_mapping, num_kv_heads,
        row_bytes / 16, block_size, num_blocks, device_status);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

int pkv_copy_blocks(void *const *k_caches, void *const *v_caches, int num_layers,
                    const int64_t *src_dst_pairs, int num_pairs, size_t block_bytes,
                    int64_t num_blocks, uint32_t *device_status, void *stream)
{
    if (num_layers < 0 || num_pairs < 0 || block_bytes == 0 || block_bytes % 16 || num_blocks <= 0)
        return PKV_EINVAL;
    if (num_layers == 0 || num_pairs == 0)
        return PKV_OK;
    if (!k_caches || !v_caches || !src_dst_pairs)
        return PKV_EINVAL;
    for (int l = 0; l < num_layers; ++l)
        if (!k_caches[l] || !v_caches[l] || !aligned16(k_caches[l]) || !aligned16(v_caches[l]))
            return PKV_EINVAL;
    for (int l0 = 0; l0 < num_layers; l0 += kCopyMaxLayers) {
        const int nl = num_layers - l0 < kCopyMaxLayers ? num_layers - l0 : kCopyMaxLayers;
        CopyBlocksParams ptrs;
        for (int l = 0; l < nl; ++l) {
            ptrs.k[l] = static_cast<uint4 *>(k_caches[l0 + l]);
            ptrs.v[l] = static_cast<uint4 *>(v_caches[l0 + l]);
        }
        dim3 grid(num_pairs, nl, 2);
        static unsigned long long copy_attr = 0;
        if (ensure_smem_attr(reinterpret_cast<const void *>(copy_blocks_kernel), 0, &copy_attr))
            return PKV_ECUDA;
        copy_blocks_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
            ptrs, src_dst_pairs, (int64_t)(block_bytes / 16), num_blocks, device_status);
        if (cudaGetLastError() != cudaSuccess)
            return PKV_ECUDA;
    }
    return PKV_OK;
}

int pkv_swap_blocks(void *const *gpu_k, void *const *gpu_v, void *const *host_k,
                    void *const *host_v, int num_layers, const int64_t *pairs, int num_pairs,
                    size_t block_bytes, int64_t gpu_blocks, int64_t host_blocks, int direction,
                    uint32_t *device_status, void *stream)
{
    if (num_layers < 0 || num_pairs < 0 || block_bytes == 0 || block_bytes % 16 ||
        gpu_blocks <= 0 || host_blocks <= 0 ||
        (direction != PKV_SWAP_OUT && direction != PKV_SWAP_IN))
        return PKV_EINVAL;
    if (num_layers == 0 || num_pairs == 0)
        return PKV_OK;
    if (!gpu_k || !gpu_v || !host_k || !host_v || !pairs)
        return PKV_EINVAL;
    for (int l0 = 0; l0 < num_layers; l0 += kSwapMaxLayers) {
        const int nl = num_layers - l0 < kSwapMaxLayers ? num_layers - l0 : kSwapMaxLayers;
        SwapBlocksParams ptrs;
        for (int l = 0; l < nl; ++l) {
            void *hk = nullptr, *hv = nullptr;
            if (!gpu_k[l0 + l] || !gpu_v[l0 + l] || !aligned16(gpu_k[l0 + l]) ||
                !aligned16(gpu_v[l0 + l]))
                return PKV_EINVAL;
            // the host pools must be pinned and mapped into the device's
            // address space (cudaHostAlloc / torch pin_memory)
            if (!host_k[l0 + l] || !host_v[l0 + l] ||
                cudaHostGetDevicePointer(&hk, host_k[l0 + l], 0) != cudaSuccess ||
                cudaHostGetDevicePointer(&hv, host_v[l0 + l], 0) != cudaSuccess ||
                !aligned16(hk) || !aligned16(hv)) {
                (void)cudaGetLastError();
                return PKV_EINVAL;
            }
            ptrs.gpu_k[l] = static_cast<uint4 *>(gpu_k[l0 + l]);
            ptrs.gpu_v[l] = static_cast<uint4 *>(gpu_v[l0 + l]);
            ptrs.host_k[l] = static_cast<uint4 *>(hk);
            ptrs.host_v[l] = static_cast<uint4 *>(hv);
        }
        static unsigned long long swap_attr = 0;
        if (ensure_smem_attr(reinterpret_cast<const void *>(swap_blocks_kernel), 0, &swap_attr))
            return PKV_ECUDA;
        dim3 grid(num_pairs, nl, 2);
        swap_blocks_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
            ptrs, pairs, (int64_t)(block_bytes / 16), gpu_blocks, host_blocks,
            direction == PKV_SWAP_OUT ? 1 : 0, device_status);
        if (cudaGetLastError() != cudaSuccess)
            return PKV_ECUDA;
    }
    return PKV_OK;
}

int pkv_test_bounded_wait(uint64_t limit_ns, uint64_t max_polls, uint32_t *device_status,
                          void *stream)
{
    if (!device_status || limit_ns == 0 || limit_ns > kWaitLimitNs)
        return PKV_EINVAL;
    bounded_wait_test_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, max_polls,
                                                                               device_status);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

}  // extern "C"
