// Device helpers shared by the kernels: streaming 16-byte memory access,
// bf16 <-> binary32 conversion and round-to-nearest adds, and bulk row copies
// through shared memory, all in inline PTX so that neither compiler flags nor
// contraction can change the arithmetic.
#pragma once

#include <stdint.h>

namespace cpt {

// ----------------------------------------------------------------- bounds checks
//
// Built with -DCPT_CHECK_BOUNDS, every index a kernel reads from memory (a
// map entry, a document boundary) or derives from one (a rank, a local row)
// is checked against the extent of the buffer it addresses before it is
// used. A failed check adds one to this translation unit's device counter
// and the access is skipped; nothing traps. Without the flag kCheckBounds is
// false and the checks compile to nothing.
#ifdef CPT_CHECK_BOUNDS
constexpr bool kCheckBounds = true;
static __device__ unsigned int g_bounds_violations;
#else
constexpr bool kCheckBounds = false;
#endif

// `ok`, counting a failure when `count` (one lane of a warp-wide check).
__device__ __forceinline__ bool in_bounds(bool ok, bool count = true)
{
#ifdef CPT_CHECK_BOUNDS
    if (!ok && count) atomicAdd(&g_bounds_violations, 1u);
    return ok;
#else
    (void)ok;
    (void)count;
    return true;
#endif
}

// This translation unit's failed-check count (0 without CPT_CHECK_BOUNDS).
static inline cudaError_t read_bounds_counter(unsigned int *count, bool reset)
{
#ifdef CPT_CHECK_BOUNDS
    cudaError_t e = cudaMemcpyFromSymbol(count, g_bounds_violations, sizeof(unsigned int));
    if (e == cudaSuccess && reset) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_bounds_violations, &zero, sizeof(unsigned int));
    }
    return e;
#else
    (void)reset;
    *count = 0;
    return cudaSuccess;
#endif
}

// 16-byte load of data read exactly once in this kernel: read-only path,
// no L1 allocation.
__device__ __forceinline__ uint4 ld_once(const void *p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// 16-byte store of data not read again by this kernel (streaming, evict-first).
__device__ __forceinline__ void st_once(void *p, uint4 v)
{
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w));
}

__device__ __forceinline__ void st_once(void *p, uint2 v)
{
    asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y));
}

// binary32 add, round to nearest even, subnormals kept, never fused.
__device__ __forceinline__ float add_rn(float a, float b)
{
    float d;
    asm("add.rn.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

// The two bf16 halves of a 32-bit word, widened exactly.
__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

// Round two binary32 values to bf16 (nearest even) and pack them, `lo` in the
// low half (the lower address in memory).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// ----------------------------------------------------------------- bulk copies
//
// Whole rows move between global and shared memory with the SM's bulk-copy
// engine (cp.async.bulk), one instruction per row; a load completes on an
// mbarrier that counts its bytes, a store is tracked as a bulk group of the
// issuing thread. Sizes and both addresses must be multiples of 16 bytes.

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t arrivals)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(arrivals));
}

// Makes initialised mbarriers visible to the bulk-copy engine.
__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrive once and announce `bytes` of bulk-copy traffic for this phase.
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{ .reg .pred q; mbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2; selp.u32 %0, 1, 0, q; }"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of `bar`, giving up after about one second of
// %globaltimer time or 2^24 polls, whichever comes first. A wait that gives up
// means a copy never completed; the caller records it and stops.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0; it < (1u << 24); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > 1000000000ull) break;
    }
    return false;
}

__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gsrc, uint32_t bytes,
                                          uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Orders this thread's generic-proxy writes to shared memory before later
// bulk copies that read it.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void bulk_store(void *gdst, const void *smem_src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
                 "r"(smem_addr(smem_src)), "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N of this thread's bulk stores still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until all of this thread's bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

}  // namespace cpt
