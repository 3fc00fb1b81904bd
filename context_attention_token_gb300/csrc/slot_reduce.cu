// Ordered one-shot sum of P slot buffers, and the bounded epoch check that
// gates it.
//
// "Add stream-ordered CP gradient return primitive" (TransformerEngine PR
// 3235), sequence diagram: after the epoch barrier each owner accumulates
// grad_key_return[0..cp_size-1] into its gradient. "Low Latency
// Communication Kernels with NVSHMEM" (GPU MODE lecture 87 notes), one-shot
// all-reduce: every element reads all P contributions in a single step. Here
// the P contributions are P buffers in one HBM; dst[i] is their binary32 sum in
// slot order, starting from slot 0's value, rounded once.
//
// Small messages are launch-latency-bound; large ones are HBM-bound. Two
// kernels share the arithmetic:
//  - slot_reduce_kernel: each thread keeps U x P 16-byte loads in flight; the
//    grid never exceeds what is resident at once, and a grid-stride loop
//    covers the rest. It handles every case and the ragged tail.
//  - slot_reduce_bulk_kernel (equal input and output types): each warp moves
//    kChunk bytes of every slot into shared memory with P bulk copies on one
//    mbarrier, sums them there, and writes the chunk back with one bulk store.
//    Whole chunks only; the rest goes to slot_reduce_kernel. Every mbarrier
//    wait has a budget; one that runs out is counted in g_wait_timeouts.
#include <atomic>

#include "cpt_device.cuh"
#include "cpt_internal.h"

namespace cpt {

namespace {

constexpr int kThreads = 256;
constexpr int kBulkWarps = 2;      // independent chunk pipelines per CTA
constexpr int kChunk = 4096;       // bytes of every slot per warp step
constexpr int kBulkMaxSmem = 112 * 1024;

// Bulk-copy waits that ran out of their budget; zero unless a copy never
// completed. Read by read_slot_reduce_wait_timeouts.
__device__ unsigned int g_wait_timeouts;

// Extra bytes announced on every bulk-copy mbarrier beyond what its copies
// deliver: 0, except while a test makes the waits run out on purpose
// (set_stall_slot_reduce).
__device__ unsigned int g_stall_tx;

template <int IN>
__device__ __forceinline__ float load_scalar(const uint8_t *base, int64_t i)
{
    if constexpr (IN == kBf16) {
        const uint16_t h = reinterpret_cast<const uint16_t *>(base)[i];
        return __uint_as_float((uint32_t)h << 16);
    } else {
        return reinterpret_cast<const float *>(base)[i];
    }
}

template <int OUT>
__device__ __forceinline__ void store_scalar(uint8_t *base, int64_t i, float v)
{
    if constexpr (OUT == kBf16) {
        const uint32_t packed = pack_bf16x2(v, 0.0f);
        reinterpret_cast<uint16_t *>(base)[i] = (uint16_t)(packed & 0xFFFFu);
    } else {
        reinterpret_cast<float *>(base)[i] = v;
    }
}

template <int IN>
__device__ __forceinline__ void widen(const uint4 &v, float (&f)[8])
{
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

__device__ __forceinline__ void widen_f32(const uint4 &v, float (&f)[4])
{
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
}

template <int P, int IN, int OUT, int U>
__global__ void __launch_bounds__(kThreads, 4) slot_reduce_kernel(const SlotReduceParams p)
{
    if (p.status != nullptr && *reinterpret_cast<const volatile int32_t *>(p.status) != 0) return;
    constexpr int E = IN == kBf16 ? 8 : 4;
    constexpr int kOutUnitBytes = E * (OUT == kBf16 ? 2 : 4);
    const int64_t n_units = p.n_elems / E;
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t nthreads = (int64_t)gridDim.x * kThreads;

    for (int64_t i0 = tid; i0 < n_units; i0 += nthreads * U) {
        uint4 v[U][P];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t i = i0 + k * nthreads;
            if (i < n_units) {
#pragma unroll
                for (int w = 0; w < P; ++w) v[k][w] = ld_once(p.s[w] + i * 16);
            }
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t i = i0 + k * nthreads;
            if (i >= n_units) continue;
            float acc[E], x[E];
            if constexpr (IN == kBf16) widen<IN>(v[k][0], acc); else widen_f32(v[k][0], acc);
#pragma unroll
            for (int w = 1; w < P; ++w) {
                if constexpr (IN == kBf16) widen<IN>(v[k][w], x); else widen_f32(v[k][w], x);
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] = add_rn(acc[e], x[e]);
            }
            uint8_t *d = p.dst + i * kOutUnitBytes;
            if constexpr (OUT == kBf16) {
                if constexpr (E == 8) {
                    st_once(d, make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                          pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7])));
                } else {
                    st_once(d, make_uint2(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3])));
                }
            } else {
#pragma unroll
                for (int h = 0; h < E; h += 4)
                    st_once(d + h * 4, make_uint4(__float_as_uint(acc[h]), __float_as_uint(acc[h + 1]),
                                                  __float_as_uint(acc[h + 2]),
                                                  __float_as_uint(acc[h + 3])));
            }
        }
    }

    // ragged tail (fewer than one 16-byte unit of elements)
    if (tid == 0) {
        for (int64_t e = n_units * E; e < p.n_elems; ++e) {
            float acc = load_scalar<IN>(p.s[0], e);
#pragma unroll
            for (int w = 1; w < P; ++w) acc = add_rn(acc, load_scalar<IN>(p.s[w], e));
            store_scalar<OUT>(p.dst, e, acc);
        }
    }
}

// dst chunk c = ordered sum of chunk c of every slot, chunks of kChunk bytes,
// equal input and output types.
template <int P, int T>
__global__ void __launch_bounds__(32 * kBulkWarps) slot_reduce_bulk_kernel(const SlotReduceParams p,
                                                                         const int64_t n_chunks)
{
    if (p.status != nullptr && *reinterpret_cast<const volatile int32_t *>(p.status) != 0) return;
    constexpr int E = T == kBf16 ? 8 : 4;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[kBulkWarps];
    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    uint8_t *stage = smem + (size_t)wid * (P + 1) * kChunk;
    uint8_t *out = stage + (size_t)P * kChunk;
    uint64_t *bar = bars + wid;
    if (lane == 0) {
        mbar_init(bar, 1);
        mbar_init_fence();
    }
    __syncwarp();
    uint32_t phase = 0;
    const uint32_t stall = g_stall_tx;
    const int64_t stride = (int64_t)gridDim.x * kBulkWarps;
    for (int64_t c = (int64_t)blockIdx.x * kBulkWarps + wid; c < n_chunks; c += stride) {
        if (lane == 0) {
            mbar_expect_tx(bar, (uint32_t)(P * kChunk) + stall);
#pragma unroll
            for (int w = 0; w < P; ++w) bulk_load(stage + (size_t)w * kChunk, p.s[w] + c * kChunk, kChunk, bar);
        }
        const bool ok = mbar_wait_bounded(bar, phase);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
            if (lane == 0) {
                atomicAdd(&g_wait_timeouts, 1u);
                mbar_wait_bounded(bar, phase);  // one more budget for the loads before leaving
            }
            break;
        }
        phase ^= 1u;
        if (lane == 0) bulk_wait_read<0>();  // the previous chunk's store has read `out`
        __syncwarp();
        for (int u = lane; u < kChunk / 16; u += 32) {
            float acc[E], x[E];
            const uint4 v0 = *reinterpret_cast<const uint4 *>(stage + (size_t)u * 16);
            if constexpr (T == kBf16) widen<T>(v0, acc); else widen_f32(v0, acc);
#pragma unroll
            for (int w = 1; w < P; ++w) {
                const uint4 v = *reinterpret_cast<const uint4 *>(stage + (size_t)w * kChunk + (size_t)u * 16);
                if constexpr (T == kBf16) widen<T>(v, x); else widen_f32(v, x);
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] = add_rn(acc[e], x[e]);
            }
            uint4 r;
            if constexpr (T == kBf16) {
                r = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                               pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
            } else {
                r = make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]), __float_as_uint(acc[2]),
                               __float_as_uint(acc[3]));
            }
            *reinterpret_cast<uint4 *>(out + (size_t)u * 16) = r;
        }
        fence_proxy_async_smem();  // the chunk's generic writes before the bulk store reads it
        __syncwarp();
        if (lane == 0) bulk_store(p.dst + c * kChunk, out, kChunk);
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
}

template <int P, int T>
cudaError_t launch_bulk(const SlotReduceParams &p, int64_t n_chunks, cudaStream_t stream)
{
    auto kernel = slot_reduce_bulk_kernel<P, T>;
    constexpr size_t smem = (size_t)kBulkWarps * (P + 1) * kChunk;
    static std::atomic<int> blocks_per_sm[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (blocks_per_sm[dev].load(std::memory_order_acquire) == 0) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, 32 * kBulkWarps, smem);
        if (e != cudaSuccess) return e;
        blocks_per_sm[dev].store(n > 0 ? n : 1, std::memory_order_release);
    }
    int64_t blocks = (int64_t)blocks_per_sm[dev].load(std::memory_order_acquire) * sm_count(dev);
    const int64_t needed = (n_chunks + kBulkWarps - 1) / kBulkWarps;
    if (blocks > needed) blocks = needed;
    kernel<<<(unsigned)blocks, 32 * kBulkWarps, smem, stream>>>(p, n_chunks);
    return cudaGetLastError();
}

// Whether the bulk kernel takes the whole chunks of this call (choice: 0 =
// measured rule, 1 = never, 2 = wherever it can run). The rule comes from the
// slot-reduce sweep on GB300 (2, 4 and 8 slots, 1 KB to 1 GB per slot, both
// kernels): right after an L2 flush the bulk kernel was 2-5 % faster at 1 GB
// per slot, even at 256 MB, and slower below (by up to 30 % on small, warm,
// back-to-back calls, where its one-chunk-per-warp pipeline shows).
constexpr int64_t kBulkMinSlotBytes = int64_t(1) << 30;

bool use_bulk(int choice, int P, int64_t bytes_per_slot)
{
    if ((int64_t)kBulkWarps * (P + 1) * kChunk > kBulkMaxSmem || bytes_per_slot < kChunk) return false;
    if (choice == 2) return true;
    return choice == 0 && bytes_per_slot >= kBulkMinSlotBytes;
}

template <int P, int IN, int OUT>
cudaError_t launch_loads(const SlotReduceParams &p, cudaStream_t stream);

template <int P, int IN, int OUT>
cudaError_t launch_typed(const SlotReduceParams &p, cudaStream_t stream)
{
    if constexpr (IN == OUT) {
        constexpr int esz = IN == kBf16 ? 2 : 4;
        const int64_t bytes = p.n_elems * esz;
        if (slot_reduce_uses_bulk(P, IN, OUT, bytes)) {
            const int64_t n_chunks = bytes / kChunk;
            cudaError_t e = launch_bulk<P, IN>(p, n_chunks, stream);
            if (e != cudaSuccess) return e;
            const int64_t done = n_chunks * kChunk;
            if (done == bytes) return cudaSuccess;
            SlotReduceParams rest = p;  // the tail after the whole chunks
            for (int w = 0; w < P; ++w) rest.s[w] = p.s[w] + done;
            rest.dst = p.dst + done;
            rest.n_elems = p.n_elems - done / esz;
            return launch_loads<P, IN, OUT>(rest, stream);
        }
    }
    return launch_loads<P, IN, OUT>(p, stream);
}

template <int P, int IN, int OUT>
cudaError_t launch_loads(const SlotReduceParams &p, cudaStream_t stream)
{
    constexpr int U = P <= 4 ? 2 : 1;
    constexpr int E = IN == kBf16 ? 8 : 4;
    auto kernel = slot_reduce_kernel<P, IN, OUT, U>;
    static std::atomic<int> blocks_per_sm[64];
    int dev = 0;
    const cudaError_t dev_err = cudaGetDevice(&dev);
    if (dev_err != cudaSuccess) return dev_err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (blocks_per_sm[dev].load(std::memory_order_acquire) == 0) {
        int n = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kThreads, 0);
        if (e != cudaSuccess) return e;
        blocks_per_sm[dev].store(n > 0 ? n : 1, std::memory_order_release);
    }
    const int64_t cap = (int64_t)blocks_per_sm[dev].load(std::memory_order_acquire) * sm_count(dev);
    const int64_t n_units = p.n_elems / E;
    int64_t blocks = (n_units + (int64_t)kThreads * U - 1) / ((int64_t)kThreads * U);
    if (blocks < 1) blocks = 1;
    if (blocks > cap) blocks = cap;
    kernel<<<(unsigned)blocks, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

template <int P>
cudaError_t launch_p(const SlotReduceParams &p, int in, int out, cudaStream_t s)
{
    if (in == kBf16 && out == kBf16) return launch_typed<P, kBf16, kBf16>(p, s);
    if (in == kBf16 && out == kF32) return launch_typed<P, kBf16, kF32>(p, s);
    if (in == kF32 && out == kBf16) return launch_typed<P, kF32, kBf16>(p, s);
    return launch_typed<P, kF32, kF32>(p, s);
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// One warp. Lane w < P watches writer w's flag. Polls until every flag has
// reached the epoch (wrap-around safe) or the time budget is spent; an
// iteration cap bounds the loop even if the timer were to stall.
__global__ void epoch_check_kernel(const uint32_t *flags_row, int P, uint32_t epoch,
                                   uint64_t timeout_ns, uint64_t max_iters, int32_t *status)
{
    const int lane = threadIdx.x;
    const uint64_t t0 = global_timer_ns();
    for (uint64_t it = 0;; ++it) {
        bool ok = true;
        if (lane < P) ok = (int32_t)(ld_acquire_gpu(flags_row + lane) - epoch) >= 0;
        if (__all_sync(0xFFFFFFFFu, ok)) {
            if (lane == 0) *status = 0;
            return;
        }
        const uint64_t elapsed = global_timer_ns() - t0;
        const bool give_up = __any_sync(0xFFFFFFFFu, elapsed >= timeout_ns || it >= max_iters);
        if (give_up) {
            if (lane == 0) *status = kStatusTimeout;
            return;
        }
        __nanosleep(512);
    }
}

}  // namespace

cudaError_t set_stall_slot_reduce(unsigned int extra_bytes)
{
    return cudaMemcpyToSymbol(g_stall_tx, &extra_bytes, sizeof(unsigned int));
}

bool slot_reduce_uses_bulk(int P, int in_dtype, int out_dtype, int64_t bytes_per_slot)
{
    return in_dtype == out_dtype && use_bulk(kernel_path(), P, bytes_per_slot);
}

cudaError_t read_slot_reduce_wait_timeouts(unsigned int *count, bool reset)
{
    cudaError_t e = cudaMemcpyFromSymbol(count, g_wait_timeouts, sizeof(unsigned int));
    if (e == cudaSuccess && reset) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_wait_timeouts, &zero, sizeof(unsigned int));
    }
    return e;
}

cudaError_t launch_slot_reduce(const SlotReduceParams &p, int n_slots, int in_dtype,
                               int out_dtype, cudaStream_t stream)
{
    if (p.n_elems == 0) return cudaSuccess;
    switch (n_slots) {
    case 1: return launch_p<1>(p, in_dtype, out_dtype, stream);
    case 2: return launch_p<2>(p, in_dtype, out_dtype, stream);
    case 3: return launch_p<3>(p, in_dtype, out_dtype, stream);
    case 4: return launch_p<4>(p, in_dtype, out_dtype, stream);
    case 5: return launch_p<5>(p, in_dtype, out_dtype, stream);
    case 6: return launch_p<6>(p, in_dtype, out_dtype, stream);
    case 7: return launch_p<7>(p, in_dtype, out_dtype, stream);
    case 8: return launch_p<8>(p, in_dtype, out_dtype, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_epoch_check(const uint32_t *flags_row, int cp_size, uint32_t epoch,
                               uint64_t timeout_ns, int32_t *status, cudaStream_t stream)
{
    // each poll costs at least one L2 round trip (hundreds of ns), so this
    // cap ends the loop within a small multiple of timeout_ns in any case
    const uint64_t max_iters = timeout_ns / 256 + 1;
    epoch_check_kernel<<<1, 32, 0, stream>>>(flags_row, cp_size, epoch, timeout_ns, max_iters,
                                             status);
    return cudaGetLastError();
}

}  // namespace cpt
