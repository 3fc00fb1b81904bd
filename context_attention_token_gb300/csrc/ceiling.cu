// Streaming ceiling for the roofline: the traffic of an HBM-bound call with
// no arithmetic and no index, moved by the SM's bulk-copy engine.
//
// dst receives a copy of srcs[0]; srcs[1..n_src) are read at the same
// offsets and discarded. With n_src = P the reads and writes are those of the
// fused gradient return (P writer rows in, one owner row out, 4:1 at P = 4);
// with n_src = 1 they are those of the row gather (1:1). One thread per CTA
// moves blocks of block_bytes through a ring of `stages` shared-memory
// stages: all n_src loads of a block complete on one mbarrier, then one bulk
// store writes the block. Every wait has a time and poll budget; a wait that
// runs out is counted in g_wait_timeouts and stops the CTA.
#include <atomic>

#include "cpt_device.cuh"
#include "cpt_internal.h"

namespace cpt {

namespace {

constexpr int kMaxStages = 8;
constexpr int kCeilingMaxSmem = 200 * 1024;

__device__ unsigned int g_wait_timeouts;

struct CeilingParams {
    const uint8_t *src[kMaxCp];
    uint8_t *dst;
    int64_t bytes;
    int32_t n_src;
    int32_t block_bytes;
    int32_t stages;
};

template <int N>
__global__ void __launch_bounds__(32) stream_ceiling_kernel(const CeilingParams p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bar[kMaxStages];
    if (threadIdx.x != 0) return;
    const int S = p.stages;
    const int64_t B = p.block_bytes;
    for (int s = 0; s < S; ++s) mbar_init(&bar[s], 1);
    mbar_init_fence();
    const int64_t nblk = (p.bytes + B - 1) / B;
    const int64_t first = blockIdx.x, step = gridDim.x;
    const int64_t mine = first < nblk ? (nblk - 1 - first) / step + 1 : 0;
    uint32_t phases = 0;

    auto stage_of = [&](int64_t i) { return smem + (size_t)(i % S) * N * B; };
    auto issue = [&](int64_t i) {
        const int64_t off = (first + i * step) * B;
        const uint32_t len = (uint32_t)min(B, p.bytes - off);
        uint8_t *st = stage_of(i);
        uint64_t *b = &bar[i % S];
        mbar_expect_tx(b, len * (uint32_t)N);
#pragma unroll
        for (int k = 0; k < N; ++k) bulk_load(st + (size_t)k * B, p.src[k] + off, len, b);
    };

    for (int64_t i = 0; i < S - 1 && i < mine; ++i) issue(i);
    for (int64_t i = 0; i < mine; ++i) {
        const int s = (int)(i % S);
        if (!mbar_wait_bounded(&bar[s], (phases >> s) & 1u)) {
            atomicAdd(&g_wait_timeouts, 1u);
            for (int64_t k = i; k < i + S - 1 && k < mine; ++k)
                mbar_wait_bounded(&bar[k % S], (phases >> (k % S)) & 1u);
            break;
        }
        phases ^= 1u << s;
        const int64_t off = (first + i * step) * B;
        bulk_store(p.dst + off, stage_of(i), (uint32_t)min(B, p.bytes - off));
        const int64_t nxt = i + S - 1;
        if (nxt < mine) {
            bulk_wait_read<1>();  // the stage of block i - 1 is free again
            issue(nxt);
        }
    }
    bulk_wait_all();
}

}  // namespace

size_t ceiling_smem_bytes(int n_src, int block_bytes, int stages)
{
    return (size_t)n_src * (size_t)block_bytes * (size_t)stages;
}

bool ceiling_shape_ok(int n_src, int block_bytes, int stages)
{
    return n_src >= 1 && n_src <= kMaxCp && stages >= 2 && stages <= kMaxStages && block_bytes >= 16 &&
           block_bytes % 16 == 0 && ceiling_smem_bytes(n_src, block_bytes, stages) <= kCeilingMaxSmem;
}

template <int N>
cudaError_t launch_n(const CeilingParams &p, int ctas_per_sm, int dev, cudaStream_t stream)
{
    static std::atomic<bool> attr_set[64];
    auto kernel = stream_ceiling_kernel<N>;
    cudaError_t e;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kCeilingMaxSmem);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_release);
    }
    const size_t smem = ceiling_smem_bytes(N, p.block_bytes, p.stages);
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 32, smem);
    if (e != cudaSuccess) return e;
    if (per_sm > ctas_per_sm) per_sm = ctas_per_sm;
    if (per_sm < 1) per_sm = 1;
    int64_t grid = (int64_t)per_sm * sm_count(dev);
    const int64_t nblk = (p.bytes + p.block_bytes - 1) / p.block_bytes;
    if (grid > nblk) grid = nblk;
    kernel<<<(unsigned)grid, 32, smem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_stream_ceiling(const uint8_t *const *srcs, int n_src, uint8_t *dst, int64_t bytes,
                                  int block_bytes, int stages, int ctas_per_sm, cudaStream_t stream)
{
    if (bytes == 0) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    CeilingParams p;
    for (int k = 0; k < kMaxCp; ++k) p.src[k] = k < n_src ? srcs[k] : nullptr;
    p.dst = dst;
    p.bytes = bytes;
    p.n_src = n_src;
    p.block_bytes = block_bytes;
    p.stages = stages;
    switch (n_src) {
    case 1: return launch_n<1>(p, ctas_per_sm, dev, stream);
    case 2: return launch_n<2>(p, ctas_per_sm, dev, stream);
    case 3: return launch_n<3>(p, ctas_per_sm, dev, stream);
    case 4: return launch_n<4>(p, ctas_per_sm, dev, stream);
    case 5: return launch_n<5>(p, ctas_per_sm, dev, stream);
    case 6: return launch_n<6>(p, ctas_per_sm, dev, stream);
    case 7: return launch_n<7>(p, ctas_per_sm, dev, stream);
    case 8: return launch_n<8>(p, ctas_per_sm, dev, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t read_ceiling_wait_timeouts(unsigned int *count, bool reset)
{
    cudaError_t e = cudaMemcpyFromSymbol(count, g_wait_timeouts, sizeof(unsigned int));
    if (e == cudaSuccess && reset) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_wait_timeouts, &zero, sizeof(unsigned int));
    }
    return e;
}

}  // namespace cpt
