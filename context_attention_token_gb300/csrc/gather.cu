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
// HBM-bound bit copy: every output row is one source row. Two kernels:
//  - gather_blocks_kernel (long rows and large launches, where it measured
//    faster: prefer_blocks; set_kernel_path overrides): the output is cut
//    into blocks of up to kBlockBytes of consecutive rows. One thread per CTA
//    moves each block through shared memory with bulk copies
//    (cp.async.bulk): source rows with consecutive indices share one bulk
//    load, destination rows of one rank piece share one bulk store, padding
//    rows are zero-filled in shared memory. A ring of kStages blocks keeps
//    loads in flight while earlier blocks are stored; the warp reads the map
//    one block ahead. Where the map is the identity, the loads ask L2 to
//    evict their lines first. Every mbarrier wait has a time and poll budget;
//    a wait that runs out is counted in g_wait_timeouts and stops the CTA.
//    Where the map is the identity and each tensor's destination is one
//    contiguous buffer (packed-contiguous partition and restore), the launch
//    is a straight copy and copy_blocks_kernel moves it in 32 KB blocks with
//    no map at all.
//  - gather_kernel (all other cases): a warp owns one row at a time and
//    moves it in 16-byte units, kUnroll units per lane in flight before the
//    first store. Rows are visited in output order by a grid-stride loop, so
//    concurrently active warps read and write neighbouring rows.
#include <atomic>

#include "cpt_device.cuh"
#include "cpt_internal.h"

namespace cpt {

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

// The blocks kernel's shape, from a sweep on GB300 (blocks of 10 to 60 KB, 2
// to 6 stages, 1 to 3 CTAs per SM; rows of 2, 4 and 5 KB, P = 4 and 8; L2
// flushed before every launch): about 40 KB per block, four stages and one
// CTA per SM was fastest or within 1 % of it at every row size, and 4 to 7 %
// faster than gather_kernel.
constexpr int kStages = 4;
constexpr int kBlockBytes = 40960;
constexpr int kMaxBlockRows = 32;  // one map entry per lane
constexpr int kBlocksMaxSmem = 200 * 1024;

// Bulk-copy waits that ran out of their budget; zero unless a copy never
// completed. Read by read_gather_wait_timeouts.
__device__ unsigned int g_wait_timeouts;

// Extra bytes announced on every bulk-copy mbarrier beyond what its copies
// deliver: 0, except while a test makes the waits run out on purpose
// (set_stall_gather).
__device__ unsigned int g_stall_tx;

// A bulk load whose lines L2 evicts first. The blocks kernel uses it where the
// map is the identity (packed-contiguous partition and restore, a straight
// copy): every block is read and rewritten at the same offset of two buffers,
// and letting the read lines go first gave 1.5 to 2.7 % on GB300 (lognormal
// batch and the pages' shape, two boxes, 8 interleaved passes). On permuted
// maps the same hint cost about 2 %, so they keep the default policy.
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void bulk_load_evict_first(void *smem_dst, const void *gsrc, uint32_t bytes,
                                                      uint64_t *bar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_addr(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}

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
        if constexpr (kCheckBounds) {
            if (!in_bounds(q >= 0 && r < p.parts, lane == 0)) continue;
        }
        const int64_t g = p.l2g ? (int64_t)__ldg(p.l2g + q) : q;
        if constexpr (kCheckBounds) {
            if (!in_bounds(g >= -1 && g < p.src_rows, lane == 0)) continue;
        }
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


// Block b of tensor t covers the launch's local rows [q0 + b*B, +n), n <= B.
// Block indices and rows stay below 2^31 (T < 2^31), so 32-bit division does.
__global__ void __launch_bounds__(32) gather_blocks_kernel(const GatherParams p, const int B)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bar[kStages];
    const int lane = threadIdx.x;
    const int64_t rb = p.row_bytes;
    const uint32_t per_t = (uint32_t)((p.T + B - 1) / B);
    const uint32_t Tp32 = (uint32_t)p.Tp;
    const int64_t nblk = (int64_t)per_t * (p.rows / p.T);
    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&bar[s], 1);
        mbar_init_fence();
    }
    __syncwarp();
    const int64_t first = blockIdx.x, step = gridDim.x;
    const int64_t mine = first < nblk ? (nblk - 1 - first) / step + 1 : 0;
    uint32_t phases = 0;  // bit s: parity of the phase stage s waits for next
    const uint32_t stall = g_stall_tx;
    const bool identity = p.l2g == nullptr;
    const uint64_t pol = l2_evict_first_policy();

    struct Blk {
        uint32_t t;
        int64_t L0;
        int n;
    };
    auto block = [&](int64_t i) {
        const uint32_t blk = (uint32_t)(first + i * step);
        Blk b;
        b.t = blk / per_t;
        b.L0 = (int64_t)(blk - b.t * per_t) * B;
        b.n = (int)min((int64_t)B, p.T - b.L0);
        return b;
    };
    // this lane's map entry for the i-th block (-2: no row)
    auto map_entry = [&](int64_t i) -> int64_t {
        if (i >= mine) return -2;
        const Blk b = block(i);
        if (lane >= b.n) return -2;
        const int64_t q = p.q0 + b.L0 + lane;
        int64_t g = p.l2g ? (int64_t)__ldg(p.l2g + q) : q;
        // an entry outside the source is not read: its row is written as zeros
        if constexpr (kCheckBounds) {
            if (!in_bounds(g >= -1 && g < p.src_rows)) g = -1;
        }
        return g;
    };
    int64_t g_ahead = map_entry(0);

    // whole warp: start the loads of the i-th block into stage i % kStages
    auto issue = [&](int64_t i) {
        const Blk b = block(i);
        const int s = (int)(i % kStages);
        uint8_t *stage = smem + (size_t)s * B * rb;
        const int64_t g = g_ahead;
        g_ahead = map_entry(i + 1);
        const int64_t g0 = __shfl_sync(0xFFFFFFFFu, g, 0);
        if (__all_sync(0xFFFFFFFFu, lane >= b.n || (g0 >= 0 && g == g0 + lane))) {
            if (lane == 0) {  // one contiguous source run
                mbar_expect_tx(&bar[s], (uint32_t)(b.n * rb) + stall);
                if (identity)
                    bulk_load_evict_first(stage, p.src[b.t] + g0 * rb, (uint32_t)(b.n * rb), &bar[s], pol);
                else
                    bulk_load(stage, p.src[b.t] + g0 * rb, (uint32_t)(b.n * rb), &bar[s]);
            }
            return;
        }
        const int real = __popc(__ballot_sync(0xFFFFFFFFu, lane < b.n && g >= 0));
        if (lane == 0) mbar_expect_tx(&bar[s], (uint32_t)(real * rb) + stall);
        int run0 = 0;
        int64_t run_g = g0;
        for (int j = 1; j <= b.n; ++j) {
            const int64_t gj = __shfl_sync(0xFFFFFFFFu, g, j & 31);
            const int64_t gp = __shfl_sync(0xFFFFFFFFu, g, j - 1);
            if (j < b.n && gp >= 0 && gj == gp + 1) continue;  // the run goes on
            if (lane == 0) {
                if (run_g >= 0) {
                    bulk_load(stage + (size_t)run0 * rb, p.src[b.t] + run_g * rb, (uint32_t)((j - run0) * rb),
                              &bar[s]);
                } else {  // a padding row (runs of padding are one row long)
                    for (int64_t u = 0; u < rb; u += 16)
                        *reinterpret_cast<uint4 *>(stage + (size_t)run0 * rb + u) = make_uint4(0, 0, 0, 0);
                    fence_proxy_async_smem();  // before the bulk store reads it
                }
            }
            run0 = j;
            run_g = gj;
        }
    };
    // lane 0: store the i-th block, one bulk store per rank piece it touches
    auto store = [&](int64_t i) {
        const Blk b = block(i);
        const uint8_t *stage = smem + (size_t)(i % kStages) * B * rb;
        int j = 0;
        while (j < b.n) {
            const uint32_t q = (uint32_t)(p.q0 + b.L0 + j);
            const uint32_t r = q / Tp32;
            const uint32_t jj = q - r * Tp32;
            if constexpr (kCheckBounds) {
                if (!in_bounds(r < (uint32_t)p.parts)) break;
            }
            const int len = (int)min((int64_t)(b.n - j), (int64_t)(Tp32 - jj));
            bulk_store(p.dst[b.t][r] + (int64_t)jj * rb, stage + (size_t)j * rb, (uint32_t)(len * rb));
            j += len;
        }
    };

    for (int64_t i = 0; i < kStages - 1 && i < mine; ++i) issue(i);
    for (int64_t i = 0; i < mine; ++i) {
        const int s = (int)(i % kStages);
        bool ok = true;
        if (lane == 0) ok = mbar_wait_bounded(&bar[s], (phases >> s) & 1u);
        if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) {
            if (lane == 0) {
                atomicAdd(&g_wait_timeouts, 1u);
                // one more budget for every block whose loads may be in flight
                for (int64_t k = i; k < i + kStages - 1 && k < mine; ++k)
                    mbar_wait_bounded(&bar[k % kStages], (phases >> (k % kStages)) & 1u);
            }
            break;
        }
        phases ^= 1u << s;
        if (lane == 0) store(i);
        const int64_t nxt = i + kStages - 1;
        if (nxt < mine) {
            // the next block reuses the stage of block i - 1, whose stores
            // are older than block i's: wait until only block i's may read
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
            issue(nxt);
        }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
}

// Identity map with one contiguous destination per tensor (the packed-contiguous
// partition and restore): a straight copy of each tensor's rows
// [q0, q0 + T), so the map and the rank pieces drop out. One thread per CTA
// moves blocks of kCopyBlockBytes through a ring of kCopyStages stages with
// one bulk load and one bulk store each. Measured on GB300 against the row-block
// gather on the same identity copies (3.2 and 8.1 GB launches, two passes):
// 6888 against 6393 GB/s and 6965 against 6435 GB/s; 8 KB blocks at two CTAs
// per SM reached 6740-6821, 16 or 64 KB blocks 6396-6803, and an L2 evict-first
// hint on the loads cost 2 %.
constexpr int kCopyStages = 3;
constexpr int kCopyBlockBytes = 32768;

__global__ void __launch_bounds__(32) copy_blocks_kernel(const GatherParams p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bar[kCopyStages];
    if (threadIdx.x != 0) return;
    for (int s = 0; s < kCopyStages; ++s) mbar_init(&bar[s], 1);
    mbar_init_fence();
    const int64_t B = kCopyBlockBytes;
    const int64_t bytes = p.T * (int64_t)p.row_bytes;   // per tensor
    const int64_t base = p.q0 * (int64_t)p.row_bytes;
    const int64_t per_t = (bytes + B - 1) / B;
    const int64_t nblk = per_t * (p.rows / p.T);
    const int64_t first = blockIdx.x, step = gridDim.x;
    const int64_t mine = first < nblk ? (nblk - 1 - first) / step + 1 : 0;
    const uint32_t stall = g_stall_tx;
    uint32_t phases = 0;  // bit s: parity of the phase stage s waits for next

    // tensor, byte offset within it and length of this CTA's i-th block
    auto where = [&](int64_t i, int &t, int64_t &off, uint32_t &len) {
        const int64_t blk = first + i * step;
        t = (int)(blk / per_t);
        off = (blk - (int64_t)t * per_t) * B;
        len = (uint32_t)min(B, bytes - off);
    };
    auto issue = [&](int64_t i) {
        int t;
        int64_t off;
        uint32_t len;
        where(i, t, off, len);
        const int s = (int)(i % kCopyStages);
        mbar_expect_tx(&bar[s], len + stall);
        bulk_load(smem + (size_t)s * B, p.src[t] + base + off, len, &bar[s]);
    };

    for (int64_t i = 0; i < kCopyStages - 1 && i < mine; ++i) issue(i);
    for (int64_t i = 0; i < mine; ++i) {
        const int s = (int)(i % kCopyStages);
        if (!mbar_wait_bounded(&bar[s], (phases >> s) & 1u)) {
            atomicAdd(&g_wait_timeouts, 1u);
            // one more budget for every block whose load may be in flight
            for (int64_t k = i; k < i + kCopyStages - 1 && k < mine; ++k)
                mbar_wait_bounded(&bar[k % kCopyStages], (phases >> (k % kCopyStages)) & 1u);
            break;
        }
        phases ^= 1u << s;
        int t;
        int64_t off;
        uint32_t len;
        where(i, t, off, len);
        bulk_store(p.dst[t][0] + base + off, smem + (size_t)s * B, len);
        const int64_t nxt = i + kCopyStages - 1;
        if (nxt < mine) {
            bulk_wait_read<1>();  // the stage of block i - 1 is free again
            issue(nxt);
        }
    }
    bulk_wait_all();
}

// The measured rule for the blocks kernel. A sweep on GB300 (partition and
// restore, rows of 1, 2 and 5 KB, launches of 25 MB to 8 GB, L2 flushed
// before each launch) found it 4-7 % faster from about 0.5 GB per launch
// with rows of 2 KB and more, even or slower on smaller launches (up to
// 13 % slower at 0.2 GB with 2 KB rows), and slower at every size with 1 KB
// rows. So: rows of at least 2 KB and launches that move at least 384 MiB.
constexpr int64_t kBlocksMinRowBytes = 2048;
constexpr int64_t kBlocksMinLaunchBytes = int64_t(384) << 20;

bool prefer_blocks(int64_t row_bytes, int64_t rows)
{
    return row_bytes >= kBlocksMinRowBytes && 2 * rows * row_bytes >= kBlocksMinLaunchBytes;
}

// Rows per block for rows of row_bytes, or 0 when the blocks kernel cannot
// take them (its stages would not fit in shared memory).
int block_rows(int64_t row_bytes)
{
    int64_t B = kBlockBytes / row_bytes;
    B = B < 1 ? 1 : (B > kMaxBlockRows ? kMaxBlockRows : B);
    return (int64_t)kStages * B * row_bytes <= kBlocksMaxSmem ? (int)B : 0;
}

// Whether the launch is a straight copy: the identity map, and every
// tensor's rank pieces laid end to end in one destination buffer.
bool is_straight_copy(const GatherParams &p)
{
    if (p.l2g != nullptr || p.parts < 1) return false;
    const int nt = (int)(p.rows / p.T);
    for (int t = 0; t < nt; ++t)
        for (int r = 1; r < p.parts; ++r)
            if (p.dst[t][r] != p.dst[t][0] + (int64_t)r * p.Tp * p.row_bytes) return false;
    return true;
}

cudaError_t launch_copy(const GatherParams &p, int dev, cudaStream_t stream)
{
    static std::atomic<bool> attr_set[64];
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        const cudaError_t e = cudaFuncSetAttribute(copy_blocks_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   kCopyStages * kCopyBlockBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_release);
    }
    const int64_t nblk = (p.T * (int64_t)p.row_bytes + kCopyBlockBytes - 1) / kCopyBlockBytes * (p.rows / p.T);
    int64_t grid = sm_count(dev);  // one CTA per SM
    if (grid > nblk) grid = nblk;
    copy_blocks_kernel<<<(unsigned)grid, 32, (size_t)kCopyStages * kCopyBlockBytes, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_blocks(const GatherParams &p, int B, int dev, cudaStream_t stream)
{
    static std::atomic<bool> attr_set[64];
    cudaError_t e;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(gather_blocks_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kBlocksMaxSmem);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_release);
    }
    const size_t smem = (size_t)kStages * B * p.row_bytes;
    const int64_t nblk = (p.T + B - 1) / B * (p.rows / p.T);
    int64_t grid = sm_count(dev);  // one CTA per SM
    if (grid > nblk) grid = nblk;
    gather_blocks_kernel<<<(unsigned)grid, 32, smem, stream>>>(p, B);
    return cudaGetLastError();
}

}  // namespace

cudaError_t set_stall_gather(unsigned int extra_bytes)
{
    return cudaMemcpyToSymbol(g_stall_tx, &extra_bytes, sizeof(unsigned int));
}

bool gather_uses_blocks(int64_t row_bytes, int64_t rows)
{
    if (block_rows(row_bytes) == 0) return false;
    const int choice = kernel_path();
    return choice == 2 || (choice == 0 && prefer_blocks(row_bytes, rows));
}

cudaError_t read_gather_bounds_violations(unsigned int *count, bool reset)
{
    return read_bounds_counter(count, reset);
}

cudaError_t read_gather_wait_timeouts(unsigned int *count, bool reset)
{
    cudaError_t e = cudaMemcpyFromSymbol(count, g_wait_timeouts, sizeof(unsigned int));
    if (e == cudaSuccess && reset) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_wait_timeouts, &zero, sizeof(unsigned int));
    }
    return e;
}

cudaError_t launch_gather(const GatherParams &p, cudaStream_t stream)
{
    if (p.rows == 0) return cudaSuccess;
    static std::atomic<int> blocks_per_sm[64];  // per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (gather_uses_blocks(p.row_bytes, p.rows))
        return is_straight_copy(p) ? launch_copy(p, dev, stream)
                                   : launch_blocks(p, block_rows(p.row_bytes), dev, stream);
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
