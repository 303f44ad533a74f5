// pkv_host.cuh -- host-side launch plumbing shared by the translation units:
// TMA descriptor encoding for a [num_blocks, Hk, bs, D] cache and the
// compile-time dispatch of the decode kernel over (head_dim, block size, G).
#pragma once

#include <cuda_runtime.h>

#include <utility>

#include "pa_cascade.cuh"
#include "pa_cascade_tc05.cuh"
#include "pa_merge.cuh"

namespace pkv {

struct DecodeLaunch {
    DecodeParams p;
    const void *k_cache;
    const void *v_cache;
    int head_dim;
    int block_size;
    int group;
    int engine;          // Engine: kEngineAuto, kEngineCudaCore or kEngineTensorCore
    bool shared;         // shared-prefix (cascade) path
    const int32_t *plan; // device copy of the cascade plan
    int num_lists;     // shared-prefix plans: CTAs per kv head
    cudaStream_t stream;
    int *engine_used;    // out: the engine that ran
};

// Encodes a 5-D TMA descriptor over one cache [NB, Hk, bs, D] (row = D * e
// bytes) whose box is one block's `box_rows` rows of one kv head, written to
// shared memory as [chunk][row][128 bytes] with 128-byte swizzling.
// Dimension order (innermost first): elements of a 128-byte chunk, row of
// the block, 128-byte chunk of the row, kv head, block.
// The box is box_rows rows of box_chunks chunks (0: all chunks of a row).
int encode_kv_map(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int elem_bytes,
                  int head_dim, int block_size, int num_kv_heads, int64_t num_blocks, int box_rows,
                  int box_chunks = 0);

// Marks a kernel as allowed to use `bytes` of dynamic shared memory on the
// current device (cached per device).
int ensure_smem_attr(const void *func, int bytes, unsigned long long *done_mask);

// Launches `kern` as a programmatic dependent of the previous kernel on the
// stream: its CTAs may become resident while that kernel drains and wait in
// griddepcontrol.wait (the shared-prefix kernels execute it before their
// first read of memory another kernel may write).
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
               Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...) == cudaSuccess ? PKV_OK
                                                                                      : PKV_ECUDA;
}

// SMs of the current device (cached per device; 152, a GB300's count, if it
// cannot be read).
inline int device_sm_count()
{
    static int cache[64] = {};
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        (void)cudaGetLastError();
        return 152;
    }
    if (cache[dev] > 0)
        return cache[dev];
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
        (void)cudaGetLastError();
        v = 152;
    }
    cache[dev] = v;
    return v;
}

int launch_decode_f32(const DecodeLaunch &a);
int launch_decode_f16(const DecodeLaunch &a);
int launch_decode_bf16(const DecodeLaunch &a);

template <typename T, int D, int BS, int G, bool TC>
int run_decode(const DecodeLaunch &a)
{
    using Sh = DecodeShape<T, D, BS, G, TC>;
    const DecodeParams &p = a.p;
    alignas(64) CUtensorMap tmk;
    alignas(64) CUtensorMap tmv;
    int rc = encode_kv_map(&tmk, a.k_cache, Elem<T>::tma, Elem<T>::bytes, D, BS, p.num_kv_heads,
                           p.num_blocks, Sh::box_rows);
    if (rc)
        return rc;
    rc = encode_kv_map(&tmv, a.v_cache, Elem<T>::tma, Elem<T>::bytes, D, BS, p.num_kv_heads,
                       p.num_blocks, Sh::box_rows);
    if (rc)
        return rc;
    static unsigned long long done = 0;
    auto kern = pa_decode_kernel<T, D, BS, G, TC>;
    rc = ensure_smem_attr(reinterpret_cast<const void *>(kern), Sh::smem, &done);
    if (rc)
        return rc;
    // The merge is a programmatic dependent of the partition pass, whose CTAs
    // allow it only as their last act: it is scheduled as the pass's last
    // wave ends, not beside its many earlier waves (an early trigger measured
    // ~3% slower on the long-context workload).
    dim3 grid(p.num_partitions, p.num_kv_heads, p.num_seqs);
    kern<<<grid, Sh::threads, Sh::smem, a.stream>>>(p, tmk, tmv);
    if (p.split) {
        static unsigned long long merge_done = 0;
        rc = ensure_smem_attr(reinterpret_cast<const void *>(pa_merge_kernel<D>), 0, &merge_done);
        if (rc)
            return rc;
        rc = launch_pdl(pa_merge_kernel<D>, dim3((unsigned)((long long)p.num_seqs * p.num_heads)),
                        dim3(kSplitMergeWarps * 32), 0, a.stream, p);
        if (rc)
            return rc;
    }
    if (a.engine_used)
        *a.engine_used = TC ? kEngineTensorCore : kEngineCudaCore;
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

// Shared-prefix (cascade) path: one CTA per (kv head, work list), then the
// merge of multi-item sequences as a programmatic dependent launch (its CTAs
// take the slots the first grid frees and wait for it to complete, so no
// launch gap separates the two).  TC05: the tcgen05 kernel (head_dim 128),
// else the warp-level MMA kernel.
template <typename T, int D, int BS, int G, bool TC05>
int run_cascade(const DecodeLaunch &a)
{
    const DecodeParams &p = a.p;
    alignas(64) CUtensorMap tmk;
    alignas(64) CUtensorMap tmv;
    int box_rows, box_chunks, smem;
    const void *kern;
    if constexpr (TC05) {
        using CC = Tc05Cfg<T, D, BS, G>;
        box_rows = CC::BOX_ROWS;
        box_chunks = 1;   // one 64-element chunk plane per load
        smem = CC::SMEM_BYTES;
        kern = reinterpret_cast<const void *>(pa_cascade_tc05_kernel<T, D, BS, G>);
    } else {
        using CC = CascadeCfg<T, D, BS, G>;
        box_rows = CC::C::BOX_ROWS;
        box_chunks = 0;
        smem = CC::SMEM_BYTES;
        kern = reinterpret_cast<const void *>(pa_cascade_kernel<T, D, BS, G>);
    }
    int rc = encode_kv_map(&tmk, a.k_cache, Elem<T>::tma, Elem<T>::bytes, D, BS, p.num_kv_heads,
                           p.num_blocks, box_rows, box_chunks);
    if (rc)
        return rc;
    rc = encode_kv_map(&tmv, a.v_cache, Elem<T>::tma, Elem<T>::bytes, D, BS, p.num_kv_heads,
                       p.num_blocks, box_rows, box_chunks);
    if (rc)
        return rc;
    static unsigned long long done = 0;
    rc = ensure_smem_attr(kern, smem, &done);
    if (rc)
        return rc;
    if constexpr (TC05) {
        // one CTA per SM, each taking every gridDim.x-th (list, kv head) unit
        const long long units = (long long)p.num_kv_heads * a.num_lists;
        const long long sms = device_sm_count();
        const unsigned ctas = (unsigned)(units < sms ? units : sms);
        rc = launch_pdl(pa_cascade_tc05_kernel<T, D, BS, G>, dim3(ctas), dim3(Tc05Cfg<T, D, BS, G>::THREADS),
                        smem, a.stream, p, tmk, tmv, a.plan, a.num_lists);
    } else {
        dim3 grid(p.num_kv_heads, a.num_lists, 1);
        rc = launch_pdl(pa_cascade_kernel<T, D, BS, G>, grid, dim3(128), smem, a.stream, p, tmk, tmv,
                        a.plan);
    }
    if (rc)
        return rc;

    static unsigned long long merge_done = 0;
    rc = ensure_smem_attr(reinterpret_cast<const void *>(pa_cascade_merge_kernel<D>), 0, &merge_done);
    if (rc)
        return rc;
    rc = launch_pdl(pa_cascade_merge_kernel<D>,
                    dim3((unsigned)(((long long)p.num_seqs * p.num_heads + 7) / 8)), dim3(128), 0,
                    a.stream, p, a.plan);
    if (rc)
        return rc;
    if (a.engine_used)
        *a.engine_used = TC05 ? kEngineTcgen05 : kEngineTensorCore;
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

// Engine choice: tensor cores for every 16-bit cache (measured faster than the
// CUDA-core engine at every G, and the only one that keeps up with HBM once
// G >= 4 query heads share a kv head); CUDA cores for fp32 caches.
// `a.engine` overrides.
template <typename T, int D, int BS, int G>
int run_engine(const DecodeLaunch &a)
{
    if constexpr (Elem<T>::bytes == 2) {
        if (a.shared) {
            // shared prefix: the warp-level MMA kernel (measured faster so
            // far), the tcgen05 one at head_dim 128 on request; per sequence:
            // warp-level MMA (a tcgen05 request included: a decode tile of <= 8
            // query rows is HBM-bound there)
            if constexpr (D == 128) {
                if (a.engine == kEngineTcgen05)
                    return run_cascade<T, D, BS, G, true>(a);
            } else {
                if (a.engine == kEngineTcgen05)
                    return PKV_EUNSUPPORTED;
            }
            return run_cascade<T, D, BS, G, false>(a);
        }
        const bool tc = a.engine != kEngineCudaCore;
        if (tc)
            return run_decode<T, D, BS, G, true>(a);
    } else {
        if (a.engine == kEngineTensorCore || a.engine == kEngineTcgen05 || a.shared)
            return PKV_EUNSUPPORTED;
    }
    return run_decode<T, D, BS, G, false>(a);
}

template <typename T, int D, int BS>
int dispatch_group(const DecodeLaunch &a)
{
    switch (a.group) {
    case 1: return run_engine<T, D, BS, 1>(a);
    case 2: return run_engine<T, D, BS, 2>(a);
    case 4: return run_engine<T, D, BS, 4>(a);
    case 8: return run_engine<T, D, BS, 8>(a);
    default: return PKV_EUNSUPPORTED;
    }
}

template <typename T, int D>
int dispatch_block(const DecodeLaunch &a)
{
    switch (a.block_size) {
    case 8: return dispatch_group<T, D, 8>(a);
    case 16: return dispatch_group<T, D, 16>(a);
    case 32: return dispatch_group<T, D, 32>(a);
    default: return PKV_EUNSUPPORTED;
    }
}

template <typename T>
int dispatch_decode(const DecodeLaunch &a)
{
    switch (a.head_dim) {
    case 64: return dispatch_block<T, 64>(a);
    case 128: return dispatch_block<T, 128>(a);
    default: return PKV_EUNSUPPORTED;
    }
}

}  // namespace pkv
