// Fused owner-gradient return: "Add stream-ordered CP gradient return
// primitive" (TransformerEngine PR 3235), "Description" and sequence diagram:
// every writer's global dK/dV goes to the owner of each token in the
// two-chunk CP layout, and the owner sums all cp_size writer slots (its own
// included). Here the scatter and the sum are one pass: the owner's row j is
// read straight from the P writers' global row l2g[o*T/P + j], summed in
// binary32 in writer order 0..P-1 starting from writer 0's value, rounded
// once, and stored. dK and dV go through the same launch.
//
// HBM-bound: per output row it reads P input rows and writes one. A warp owns
// one output row at a time; each lane keeps kUnroll x P 16-byte loads in
// flight before summing, and the grid is a whole number of CTAs per SM, each
// warp striding over rows in output order.
#include "cpt_device.cuh"
#include "cpt_internal.h"

namespace cpt {

namespace {

constexpr int kThreads = 256;

// Elements of one 16-byte input unit, widened to binary32.
template <int IN>
struct Unit;

template <>
struct Unit<kBf16> {
    static constexpr int kElems = 8;
    __device__ __forceinline__ static void widen(const uint4 &v, float (&f)[8])
    {
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
        f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
        f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
        f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    }
};

template <>
struct Unit<kF32> {
    static constexpr int kElems = 4;
    __device__ __forceinline__ static void widen(const uint4 &v, float (&f)[4])
    {
        f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
    }
};

// Round (bf16) or keep (f32) kElems sums and store them at p.
template <int OUT, int E>
__device__ __forceinline__ void store_unit(uint8_t *p, const float (&a)[E])
{
    if constexpr (OUT == kBf16) {
        if constexpr (E == 8) {
            st_once(p, make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]),
                                  pack_bf16x2(a[4], a[5]), pack_bf16x2(a[6], a[7])));
        } else {
            st_once(p, make_uint2(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3])));
        }
    } else {
        st_once(p, make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                              __float_as_uint(a[3])));
        if constexpr (E == 8) {
            st_once(p + 16, make_uint4(__float_as_uint(a[4]), __float_as_uint(a[5]),
                                       __float_as_uint(a[6]), __float_as_uint(a[7])));
        }
    }
}

// Widen the current owner values of one unit (ACC mode). A coherent
// streaming load: this thread overwrites the same bytes afterwards.
template <int OUT, int E>
__device__ __forceinline__ void load_unit(const uint8_t *p, float (&a)[E])
{
    if constexpr (OUT == kBf16) {
        if constexpr (E == 8) {
            const uint4 v = __ldcs(reinterpret_cast<const uint4 *>(p));
            a[0] = bf16_lo(v.x); a[1] = bf16_hi(v.x); a[2] = bf16_lo(v.y); a[3] = bf16_hi(v.y);
            a[4] = bf16_lo(v.z); a[5] = bf16_hi(v.z); a[6] = bf16_lo(v.w); a[7] = bf16_hi(v.w);
        } else {
            const uint2 v = __ldcs(reinterpret_cast<const uint2 *>(p));
            a[0] = bf16_lo(v.x); a[1] = bf16_hi(v.x); a[2] = bf16_lo(v.y); a[3] = bf16_hi(v.y);
        }
    } else {
#pragma unroll
        for (int h = 0; h < E; h += 4) {
            const uint4 v = __ldcs(reinterpret_cast<const uint4 *>(p + h * 4));
            a[h] = __uint_as_float(v.x); a[h + 1] = __uint_as_float(v.y);
            a[h + 2] = __uint_as_float(v.z); a[h + 3] = __uint_as_float(v.w);
        }
    }
}

// ACC = false: out = round(x_0 + x_1 + ... + x_{P-1}), accumulator from x_0.
// ACC = true:  out = round(out + x_0 + ... + x_{P-1}), accumulator from out.
template <int P, int IN, int OUT, int U, bool ACC>
__global__ void __launch_bounds__(kThreads) grad_return_kernel(const GradReturnParams p)
{
    constexpr int E = Unit<IN>::kElems;
    constexpr int kOutUnitBytes = E * (OUT == kBf16 ? 2 : 4);
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
    const int units = p.units;

    for (int64_t R = warp; R < p.rows; R += nwarps) {
        const int t = R >= p.T;
        const int64_t q = p.q0 + (R - t * p.T);
        const int o = (int)(q / p.Tp);
        const int64_t j = q - (int64_t)o * p.Tp;
        const int64_t g = __ldg(p.l2g + q);
        const uint8_t *src[P];
#pragma unroll
        for (int w = 0; w < P; ++w) src[w] = (t ? p.w[1][w] : p.w[0][w]) + g * p.in_row_bytes;
        uint8_t *dst = (t ? p.o[1][o] : p.o[0][o]) + j * p.out_row_bytes;

        for (int u0 = lane; u0 < units; u0 += 32 * U) {
            uint4 v[U][P];
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int u = u0 + 32 * k;
                if (u < units) {
#pragma unroll
                    for (int w = 0; w < P; ++w) v[k][w] = ld_once(src[w] + (int64_t)u * 16);
                }
            }
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int u = u0 + 32 * k;
                if (u < units) {
                    uint8_t *out = dst + (int64_t)u * kOutUnitBytes;
                    float acc[E];
                    if constexpr (ACC) {
                        load_unit<OUT>(out, acc);
                    } else {
                        Unit<IN>::widen(v[k][0], acc);
                    }
#pragma unroll
                    for (int w = ACC ? 0 : 1; w < P; ++w) {
                        float x[E];
                        Unit<IN>::widen(v[k][w], x);
#pragma unroll
                        for (int e = 0; e < E; ++e) acc[e] = add_rn(acc[e], x[e]);
                    }
                    store_unit<OUT>(out, acc);
                }
            }
        }
    }
}

template <int P, int IN, int OUT, bool ACC>
cudaError_t launch_typed(const GradReturnParams &p, cudaStream_t stream)
{
    constexpr int U = P <= 4 ? 2 : 1;
    auto kernel = grad_return_kernel<P, IN, OUT, U, ACC>;
    static int blocks_per_sm[64] = {0};  // per device, one table per instantiation
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
    int64_t blocks = (p.rows + (kThreads / 32) - 1) / (kThreads / 32);
    if (blocks > cap) blocks = cap;
    kernel<<<(unsigned)blocks, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

template <int P, bool ACC>
cudaError_t launch_p(const GradReturnParams &p, int in, int out, cudaStream_t s)
{
    if (in == kBf16 && out == kBf16) return launch_typed<P, kBf16, kBf16, ACC>(p, s);
    if (in == kBf16 && out == kF32) return launch_typed<P, kBf16, kF32, ACC>(p, s);
    if (in == kF32 && out == kBf16) return launch_typed<P, kF32, kBf16, ACC>(p, s);
    return launch_typed<P, kF32, kF32, ACC>(p, s);
}

template <bool ACC>
cudaError_t launch_acc(const GradReturnParams &p, int cp_size, int in, int out, cudaStream_t s)
{
    switch (cp_size) {
    case 1: return launch_p<1, ACC>(p, in, out, s);
    case 2: return launch_p<2, ACC>(p, in, out, s);
    case 3: return launch_p<3, ACC>(p, in, out, s);
    case 4: return launch_p<4, ACC>(p, in, out, s);
    case 5: return launch_p<5, ACC>(p, in, out, s);
    case 6: return launch_p<6, ACC>(p, in, out, s);
    case 7: return launch_p<7, ACC>(p, in, out, s);
    case 8: return launch_p<8, ACC>(p, in, out, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_grad_return(const GradReturnParams &p, int cp_size, int in_dtype,
                               int out_dtype, cudaStream_t stream, bool accumulate)
{
    if (p.rows == 0) return cudaSuccess;
    return accumulate ? launch_acc<true>(p, cp_size, in_dtype, out_dtype, stream)
                      : launch_acc<false>(p, cp_size, in_dtype, out_dtype, stream);
}

}  // namespace cpt
