// Row gather between global and rank-local token order, used three ways:
//  - the Q/K/V reorder of "[PyTorch] Add experimental packed-contiguous THD
//    all-gather CP" (TransformerEngine PR 3221, commit "Reuse the existing THD
//    CUDA partition and reorder kernels ..."): index = l2g;
//  - its inverse after an all-gather, back to global order: index = g2l;
//  - the per-writer scatter into owner slots of "Add stream-ordered CP
//    gradient return primitive" (TransformerEngine PR 3235, sequence diagram):
//    index = l2g, one destination pointer per owner;
//  - the padded layout: index -1 marks a padding row, written as zeros.
//
// HBM-bound bit copy: every output row is one source row. A warp owns one row
// at a time and moves it in 16-byte units, kUnroll units per lane in flight
// before the first store. Rows are visited in output order by a grid-stride
// loop, so concurrently active warps read and write neighbouring rows.
#include <atomic>

#include "cpt_device.cuh"
#include "cpt_internal.h"

namespace cpt {

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kThreads) gather_kernel(const GatherParams p)
{
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
    const int units = p.units;

    for (int64_t R = warp; R < p.rows; R += nwarps) {
        const int t = (R >= p.T) + (R >= 2 * p.T);
        const int64_t q = p.q0 + (R - t * p.T);
        const int r = (int)(q / p.Tp);
        const int64_t j = q - (int64_t)r * p.Tp;
        const int64_t g = p.l2g ? (int64_t)__ldg(p.l2g + q) : q;
        uint8_t *dst = p.dst[t][r] + j * p.row_bytes;
        if (g < 0) {  // padding row of the padded layout
            for (int u = lane; u < units; u += 32) st_once(dst + (int64_t)u * 16, make_uint4(0, 0, 0, 0));
            continue;
        }
        const uint8_t *src = p.src[t] + g * p.row_bytes;

        for (int u0 = lane; u0 < units; u0 += 32 * kUnroll) {
            uint4 v[kUnroll];
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const int u = u0 + 32 * k;
                if (u < units) v[k] = ld_once(src + (int64_t)u * 16);
            }
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const int u = u0 + 32 * k;
                if (u < units) st_once(dst + (int64_t)u * 16, v[k]);
            }
        }
    }
}

}  // namespace

cudaError_t launch_gather(const GatherParams &p, cudaStream_t stream)
{
    if (p.rows == 0) return cudaSuccess;
    static std::atomic<int> blocks_per_sm[64];  // per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (blocks_per_sm[dev].load(std::memory_order_acquire) == 0) {
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gather_kernel, kThreads, 0);
        if (e != cudaSuccess) return e;
        blocks_per_sm[dev].store(per_sm > 0 ? per_sm : 1, std::memory_order_release);
    }
    const int64_t cap = (int64_t)blocks_per_sm[dev].load(std::memory_order_acquire) * sm_count(dev);
    int64_t blocks = (p.rows + (kThreads / 32) - 1) / (kThreads / 32);  // one warp per row
    if (blocks > cap) blocks = cap;
    gather_kernel<<<(unsigned)blocks, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace cpt
