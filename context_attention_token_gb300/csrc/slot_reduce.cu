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
// Small messages are launch-latency-bound; large ones are HBM-bound: each
// thread keeps U x P 16-byte loads in flight; the grid never exceeds what is
// resident at once, and a grid-stride loop covers the rest.
#include "cpt_device.cuh"
#include "cpt_internal.h"

namespace cpt {

namespace {

constexpr int kThreads = 256;

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

template <int P, int IN, int OUT>
cudaError_t launch_typed(const SlotReduceParams &p, cudaStream_t stream)
{
    constexpr int U = P <= 4 ? 2 : 1;
    constexpr int E = IN == kBf16 ? 8 : 4;
    auto kernel = slot_reduce_kernel<P, IN, OUT, U>;
    static int blocks_per_sm[64] = {0};
    int dev = 0;
    const cudaError_t dev_err = cudaGetDevice(&dev);
    if (dev_err != cudaSuccess) return dev_err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (blocks_per_sm[dev] == 0) {
        int n = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kThreads, 0);
        if (e != cudaSuccess) return e;
        blocks_per_sm[dev] = n > 0 ? n : 1;
    }
    const int64_t cap = (int64_t)blocks_per_sm[dev] * sm_count(dev);
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

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
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
