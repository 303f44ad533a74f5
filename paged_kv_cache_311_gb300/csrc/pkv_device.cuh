// pkv_device.cuh -- device-side building blocks for sm_103a: mbarrier and
// TMA (cp.async.bulk.tensor) wrappers in inline PTX, bounded waits, element
// conversions and packed fp32x2 arithmetic.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <type_traits>

#include "../../include/pkv.h"

namespace pkv {

// ------------------------------------------------------------ smem address
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Makes mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// One plain arrival on the barrier (release: this thread's earlier writes are
// visible to a thread that sees the phase complete).
__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of the phase (mbarrier.try_wait may suspend the thread
// for a while; an event loop that watches several barriers must not).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Limit of every wait on a load or a tensor-core product (and of the drain
// that follows a wait that gave up): 2 s of %globaltimer time.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Waits until the barrier's phase with the given parity has completed.
// Gives up and returns false after `limit_ns` of wall time or `max_polls`
// polls of the barrier, whichever comes first (0: one poll per 4 ns of the
// limit; a poll takes longer than that, so the time limit decides unless the
// timer stalls); the caller then reports PKV_DEV_TIMEOUT instead of spinning
// forever.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs,
                                                  uint64_t max_polls = 0)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t cap = max_polls ? max_polls : limit_ns >> 2;
    const uint64_t t0 = globaltimer_ns();
    for (uint64_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((it & 255u) == 0 && (globaltimer_ns() - t0 > limit_ns || it >= cap))
            return false;
    }
}

__device__ __forceinline__ void report(uint32_t *status, uint32_t bits);

// After a wait gave up: waits (bounded as any wait) for a phase whose copies
// or products were already issued, so that the CTA does not leave with them
// still writing into its shared memory or tensor memory.  If this wait gives
// up too, PKV_DEV_DRAIN_TIMEOUT reports that the CTA may have exited with
// them in flight.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity, uint32_t *status,
                                           uint64_t limit_ns = kWaitLimitNs, uint64_t max_polls = 0)
{
    if (!mbar_wait_bounded(bar, parity, limit_ns, max_polls))
        report(status, PKV_DEV_DRAIN_TIMEOUT);
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// its later async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ TMA
// 5-D tiled tensor load global -> shared with mbarrier byte accounting.
__device__ __forceinline__ void tma_load_5d(void *dst_smem, const CUtensorMap *map,
                                            uint64_t *bar, int c0, int c1, int c2, int c3, int c4)
{
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst_smem)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
        "r"(c3), "r"(c4)
        : "memory");
}

// 4-byte asynchronous copy global -> shared (no register staging); complete
// the thread's copies with cp_async_wait_all before reading them.
__device__ __forceinline__ void cp_async4(void *dst_smem, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst_smem)), "l"(src)
                 : "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------- shared loads
__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ float4 lds128f(uint32_t addr)
{
    uint4 v = lds128(addr);
    return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                       __uint_as_float(v.w));
}

__device__ __forceinline__ float2 lds64f(uint32_t addr)
{
    uint2 v = lds64(addr);
    return make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
}

// ------------------------------------------------------ element types
template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int bytes = 4;
    static constexpr CUtensorMapDataType tma = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
};
template <> struct Elem<__half> {
    static constexpr int bytes = 2;
    static constexpr CUtensorMapDataType tma = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
};
template <> struct Elem<__nv_bfloat16> {
    static constexpr int bytes = 2;
    static constexpr CUtensorMapDataType tma = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
};

// One 32-bit word of storage -> fp32 values.  For 16-bit types the word holds
// two consecutive elements (lower address in the low half).
template <typename T> struct Unpack;
template <> struct Unpack<__nv_bfloat16> {
    // bf16 is the top half of an fp32: the conversion is exact bit placement.
    __device__ __forceinline__ static float2 pair(uint32_t w)
    {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
};
template <> struct Unpack<__half> {
    __device__ __forceinline__ static float2 pair(uint32_t w)
    {
        __half2 h = *reinterpret_cast<__half2 *>(&w);
        return __half22float2(h);
    }
};

__device__ __forceinline__ float to_float(float x) { return x; }
__device__ __forceinline__ float to_float(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }

// ------------------------------------------------ packed fp32x2 arithmetic
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c)
{
    return __ffma2_rn(a, b, c);
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) { return __fmul2_rn(a, b); }

// -------------------------------------------------------- status reporting
__device__ __forceinline__ void report(uint32_t *status, uint32_t bits)
{
    if (status)
        atomicOr(status, bits);
}

}  // namespace pkv

namespace pkv {

// ------------------------------------------------- warp-level tensor cores
// ldmatrix: four 8x8 b16 matrices; lanes 8j..8j+7 give the row addresses of
// matrix j, and register j of every lane receives its fragment of matrix j.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// Transpose of an 8x8 b16 matrix held one row pair per lane.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a)
{
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

// D = A * B + D, m16n8k16, fp32 accumulators.
template <typename T> struct Mma;
template <> struct Mma<__nv_bfloat16> {
    __device__ __forceinline__ static void run(float (&c)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1)
    {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    // (lo, hi) fp32 -> one b32 of two bf16 (round to nearest even), and back.
    __device__ __forceinline__ static uint32_t pack(float lo, float hi)
    {
        uint32_t d;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
        return d;
    }
    __device__ __forceinline__ static float2 unpack(uint32_t w) { return Unpack<__nv_bfloat16>::pair(w); }
};
template <> struct Mma<__half> {
    __device__ __forceinline__ static void run(float (&c)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1)
    {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    __device__ __forceinline__ static uint32_t pack(float lo, float hi)
    {
        uint32_t d;
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
        return d;
    }
    __device__ __forceinline__ static float2 unpack(uint32_t w) { return Unpack<__half>::pair(w); }
};

}  // namespace pkv

namespace pkv {
namespace tc05 {

// ------------------------------------------- 5th-generation tensor cores
// Shared-memory matrix descriptor with 128-byte swizzling (the layout the
// TMA's 128-byte swizzle writes: 8-row atoms of 128-byte rows, 16-byte
// pieces of row r at piece ^ (r % 8); atoms 1024-byte aligned).  K-major
// operands: sbo = byte stride between 8-row groups, lbo unused; MN-major
// operands: lbo = byte stride between 64-element chunks along M (or N), sbo
// = byte stride between 8-row groups along K.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((addr >> 4) & 0x3fffu) | (uint64_t)((lbo >> 4) & 0x3fffu) << 16 |
           (uint64_t)((sbo >> 4) & 0x3fffu) << 32 | (uint64_t)1 << 46 | (uint64_t)2 << 61;
}

// Instruction descriptor of kind::f16 with fp32 accumulation: A and B of
// the cache's 16-bit type, M x N, each operand K-major or MN-major.
template <typename T>
__device__ __forceinline__ uint32_t idesc(int M, int N, bool a_mn, bool b_mn)
{
    constexpr uint32_t fmt = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
    return 1u << 4 | fmt << 7 | fmt << 10 | (a_mn ? 1u : 0u) << 15 | (b_mn ? 1u : 0u) << 16 |
           (uint32_t)(N >> 3) << 17 | (uint32_t)(M >> 4) << 24;
}

// D (TMEM) = A * B (+ D when acc), issued by one thread.
__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, bool acc)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "l"(a), "l"(b), "r"(id), "r"(acc ? 1u : 0u)
                 : "memory");
}

// The barrier's next phase completes when every MMA this thread issued so
// far has completed.
__device__ __forceinline__ void commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// Warp-collective TMEM allocation of `ncols` columns (a power of two >= 32);
// the address is written to *slot.
__device__ __forceinline__ void alloc(uint32_t *slot, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Ordering of tensor-core operations across a thread barrier.
__device__ __forceinline__ void fence_before_sync()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Warp-collective: this warp's 32 TMEM lanes (lane quarter warp % 4), 8
// consecutive 32-bit columns from `taddr` (lane field included): thread t
// receives lane (base + t).
__device__ __forceinline__ void ld8(uint32_t taddr, uint32_t (&r)[8])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7])
                 : "r"(taddr));
}
__device__ __forceinline__ void st8(uint32_t taddr, const uint32_t (&r)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}
// 32 consecutive columns of this warp's 32 lanes: thread t receives lane
// (base + t), one register per column.
__device__ __forceinline__ void ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
                 "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
                 "%28, %29, %30, %31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
                   "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
                   "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
                   "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
                   "=r"(r[31])
                 : "r"(taddr));
}
__device__ __forceinline__ void st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
                 "%10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, "
                 "%27, %28, %29, %30, %31, %32};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
                 "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
                 "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
                 "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
                 "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
}
__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

}  // namespace tc05
}  // namespace pkv
