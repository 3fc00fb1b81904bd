// Device helpers shared by the kernels: streaming 16-byte memory access,
// bf16 <-> binary32 conversion and round-to-nearest adds, in inline PTX so
// that neither compiler flags nor contraction can change the arithmetic.
#pragma once

#include <stdint.h>

namespace cpt {

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

}  // namespace cpt
