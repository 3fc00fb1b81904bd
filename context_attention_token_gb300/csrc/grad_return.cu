// Fused owner-gradient return: "Add stream-ordered CP gradient return
// primitive" (TransformerEngine PR 3235), "Description" and sequence diagram:
// every writer's global dK/dV goes to the owner of each token in the
// two-chunk CP layout, and the owner sums all cp_size writer slots (its own
// included). Here the scatter and the sum are one pass: the owner's row j is
// read straight from the P writers' global row l2g[o*T/P + j], summed in
// binary32 in writer order 0..P-1 starting from writer 0's value, rounded
// once, and stored. dK and dV go through the same launch.
//
// HBM-bound: per output row it reads P input rows and writes one. Two kernels
// share the arithmetic (binary32 adds in writer order):
//  - grad_return_bulk_kernel, in the cp_size, row and launch sizes where it
//    measured faster (prefer_bulk; set_kernel_path overrides the rule), for
//    any input and output types and either mode. Every warp runs its
//    own row pipeline: lane 0 brings the P writer rows into shared memory
//    with P bulk copies (cp.async.bulk) counted on one mbarrier, the warp
//    sums them out of shared memory into a staged output row, and lane 0
//    writes that row back with one bulk store. Every mbarrier wait has a
//    time and poll budget; a wait that runs out is counted in
//    g_wait_timeouts and stops the warp.
//  - grad_return_kernel, for all other cases (short rows, small launches,
//    P <= 2): a warp owns one output row at a time and each lane keeps
//    U x P 16-byte loads in flight before summing.
// Both size the grid to whole CTAs per SM and stride over rows in output order.
#include <atomic>

#include "cpt_device.cuh"
#include "cpt_internal.h"

namespace cpt {

namespace {

constexpr int kThreads = 256;
constexpr int kBulkWarps = 2;                 // independent row pipelines per CTA
constexpr int kBulkMaxSmem = 112 * 1024;      // keeps two CTAs (four warps) on every SM

// Where the bulk-copy kernel beats the 16-byte-load one, from a sweep on
// GB300 (P = 1..8, rows of 1 to 8 KB, bf16 and float32, 4 GB of writer rows
// per launch, two passes): it wins by 2 to 9 % from P = 5 up at every row
// size, for bf16 rows of 2 KB and more at P = 4 and 3 KB and more at P = 3,
// and for float32 rows up to 2 KB at P = 4. It loses at P = 1 and 2, and by
// about 20 % wherever its shared memory leaves one CTA per SM.
//
// With L2 flushed before every launch (as after an attention backward that
// has just written the writer rows), the bulk kernel also starts more
// slowly. At P = 4 and 6 it lost 1-7 % on launches of 0.17 to 1.3 GB. At
// 2.7 GB it tied at P = 4 and won by 1.5 % at P = 6; at 5.4 GB it won by
// 1-2 % at P = 4 and 4.5 % at P = 6. At P = 8 it won at almost every size.
// So for P <= 6 the rule also asks for launches of at least 2 GiB.
constexpr int64_t kBulkMinLaunchBytes = int64_t(2) << 30;

// Whether the bulk kernel can take rows of these sizes: its stages fit the
// shared-memory budget, and the output rows (half the input row for float32
// in, bf16 out) stay whole 16-byte units, as bulk copies need.
bool bulk_fits(int P, int64_t row_bytes, int64_t out_row_bytes)
{
    return out_row_bytes % 16 == 0 && (int64_t)kBulkWarps * (P * row_bytes + out_row_bytes) <= kBulkMaxSmem;
}

bool prefer_bulk(int P, int type, int64_t row_bytes, int64_t out_row_bytes, int64_t launch_bytes)
{
    if (row_bytes < 1024 || !bulk_fits(P, row_bytes, out_row_bytes)) return false;
    if (P <= 6 && launch_bytes < kBulkMinLaunchBytes) return false;
    if (P >= 5) return true;
    if (P == 4) return type == kBf16 ? row_bytes >= 2048 : row_bytes <= 2048;
    if (P == 3) return type == kBf16 && row_bytes >= 3072;
    return false;
}

// 0 = the measured rule, 1 = always the 16-byte-load kernel, 2 = the bulk
// kernel wherever it can run (set_kernel_path).
std::atomic<int> g_kernel_choice{0};

// Bulk-copy waits that ran out of their budget (see mbar_wait_bounded); zero
// unless a copy never completed. Read and reset by read_wait_timeouts.
__device__ unsigned int g_wait_timeouts;

// Extra bytes announced on every bulk-copy mbarrier beyond what its copies
// deliver: 0, except while a test makes the waits run out on purpose
// (set_stall_grad_return).
__device__ unsigned int g_stall_tx;

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

// The current owner values of one unit (ACC mode), loaded raw so that the
// load can be issued with the writer loads and widened after they land:
// E output elements, 8, 16 or 32 bytes. Coherent streaming loads: this
// thread overwrites the same bytes afterwards.
template <int OUT, int E>
struct OwnerUnit {
    uint4 r[(E * (OUT == kBf16 ? 2 : 4) + 15) / 16];
};

template <int OUT, int E>
__device__ __forceinline__ void load_owner(const uint8_t *p, OwnerUnit<OUT, E> &o)
{
    if constexpr (OUT == kBf16 && E == 4) {
        const uint2 v = __ldcs(reinterpret_cast<const uint2 *>(p));
        o.r[0] = make_uint4(v.x, v.y, 0u, 0u);
    } else {
#pragma unroll
        for (int h = 0; h < (int)(sizeof(o.r) / 16); ++h) o.r[h] = __ldcs(reinterpret_cast<const uint4 *>(p) + h);
    }
}

template <int OUT, int E>
__device__ __forceinline__ void widen_owner(const OwnerUnit<OUT, E> &o, float (&a)[E])
{
    if constexpr (OUT == kBf16) {
        const uint32_t w[4] = {o.r[0].x, o.r[0].y, o.r[0].z, o.r[0].w};
#pragma unroll
        for (int h = 0; h < E / 2; ++h) {
            a[2 * h] = bf16_lo(w[h]);
            a[2 * h + 1] = bf16_hi(w[h]);
        }
    } else {
#pragma unroll
        for (int h = 0; h < E / 4; ++h) {
            a[4 * h] = __uint_as_float(o.r[h].x); a[4 * h + 1] = __uint_as_float(o.r[h].y);
            a[4 * h + 2] = __uint_as_float(o.r[h].z); a[4 * h + 3] = __uint_as_float(o.r[h].w);
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
        if constexpr (kCheckBounds) {
            if (!in_bounds(q >= 0 && o < P, lane == 0)) continue;
        }
        const int64_t g = __ldg(p.l2g + q);
        if constexpr (kCheckBounds) {
            if (!in_bounds(g >= 0 && g < p.w_rows, lane == 0)) continue;
        }
        const uint8_t *src[P];
#pragma unroll
        for (int w = 0; w < P; ++w) src[w] = (t ? p.w[1][w] : p.w[0][w]) + g * p.in_row_bytes;
        uint8_t *dst = (t ? p.o[1][o] : p.o[0][o]) + j * p.out_row_bytes;

        for (int u0 = lane; u0 < units; u0 += 32 * U) {
            uint4 v[U][P];
            OwnerUnit<OUT, E> own[U];
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int u = u0 + 32 * k;
                if (u < units) {
#pragma unroll
                    for (int w = 0; w < P; ++w) v[k][w] = ld_once(src[w] + (int64_t)u * 16);
                    if constexpr (ACC) load_owner<OUT, E>(dst + (int64_t)u * kOutUnitBytes, own[k]);
                }
            }
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int u = u0 + 32 * k;
                if (u < units) {
                    uint8_t *out = dst + (int64_t)u * kOutUnitBytes;
                    float acc[E];
                    if constexpr (ACC) {
                        widen_owner<OUT, E>(own[k], acc);
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

// One output unit (the E elements of a 16-byte input unit) in shared memory:
// read back as binary32, or written from binary32 with one rounding for bf16.
template <int OUT, int E>
__device__ __forceinline__ void widen_out(const uint8_t *p, float (&a)[E])
{
    if constexpr (OUT == kBf16) {
        const uint32_t *w = reinterpret_cast<const uint32_t *>(p);
#pragma unroll
        for (int h = 0; h < E / 2; ++h) {
            a[2 * h] = bf16_lo(w[h]);
            a[2 * h + 1] = bf16_hi(w[h]);
        }
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e) a[e] = reinterpret_cast<const float *>(p)[e];
    }
}

template <int OUT, int E>
__device__ __forceinline__ void pack_out(uint8_t *p, const float (&a)[E])
{
    if constexpr (OUT == kBf16) {
        uint32_t *w = reinterpret_cast<uint32_t *>(p);
#pragma unroll
        for (int h = 0; h < E / 2; ++h) w[h] = pack_bf16x2(a[2 * h], a[2 * h + 1]);
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e) reinterpret_cast<float *>(p)[e] = a[e];
    }
}

// Any input and output types, either mode, through shared memory. Per warp:
// a stage of P input rows and one output row (which holds the owner's current
// row in accumulate mode). Lane 0 issues the loads of a row while the map
// entry of the row after it is already being fetched.
template <int P, int IN, int OUT, bool ACC>
__global__ void __launch_bounds__(32 * kBulkWarps) grad_return_bulk_kernel(const GradReturnParams p)
{
    constexpr int E = Unit<IN>::kElems;
    constexpr int kOutUnitBytes = E * (OUT == kBf16 ? 2 : 4);
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[kBulkWarps];
    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    const int rb = p.in_row_bytes;
    const int ob = p.out_row_bytes;
    uint8_t *stage = smem + (size_t)wid * ((size_t)P * rb + ob);
    uint8_t *out = stage + (size_t)P * rb;
    uint64_t *bar = bars + wid;
    if (lane == 0) {
        mbar_init(bar, 1);
        mbar_init_fence();
    }
    __syncwarp();
    const int64_t stride = (int64_t)gridDim.x * kBulkWarps;
    int64_t R = (int64_t)blockIdx.x * kBulkWarps + wid;
    int64_t g_next = 0;
    const uint32_t stall = g_stall_tx;
    // the map entry of local row q, or -1 (which fails the row's check) for a
    // row outside the map in a bounds-checked build
    auto map_at = [&](int64_t q) -> int64_t {
        if constexpr (kCheckBounds) {
            if (!in_bounds(q >= 0 && q < (int64_t)P * p.Tp)) return -1;
        }
        return __ldg(p.l2g + q);
    };
    if (lane == 0 && R < p.rows) g_next = map_at(p.q0 + (R >= p.T ? R - p.T : R));
    uint32_t phase = 0;

    for (; R < p.rows; R += stride) {
        const int t = R >= p.T;
        const int64_t q = p.q0 + (R - t * p.T);
        const int o = (int)(q / p.Tp);
        const int64_t j = q - (int64_t)o * p.Tp;
        bool row_ok = true;
        if (lane == 0) {
            const int64_t g = g_next;
            if constexpr (kCheckBounds) row_ok = in_bounds(o < P && g >= 0 && g < p.w_rows);
            if (row_ok) {
                // accumulate mode reloads `out` with the owner's current row:
                // the previous row's store must have read it first
                if constexpr (ACC) bulk_wait_read<0>();
                mbar_expect_tx(bar, (uint32_t)(P * rb + (ACC ? ob : 0)) + stall);
#pragma unroll
                for (int w = 0; w < P; ++w)
                    bulk_load(stage + (size_t)w * rb, (t ? p.w[1][w] : p.w[0][w]) + g * rb,
                              (uint32_t)rb, bar);
                if constexpr (ACC)
                    bulk_load(out, (t ? p.o[1][o] : p.o[0][o]) + j * ob, (uint32_t)ob, bar);
            }
            const int64_t Rn = R + stride;
            if (Rn < p.rows) g_next = map_at(p.q0 + (Rn >= p.T ? Rn - p.T : Rn));
        }
        if constexpr (kCheckBounds) {
            if (!__shfl_sync(0xFFFFFFFFu, row_ok, 0)) continue;  // a skipped row: nothing in flight
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
        if (!ACC && lane == 0) bulk_wait_read<0>();  // the previous row's store has read `out`
        __syncwarp();
        for (int u = lane; u < p.units; u += 32) {
            uint8_t *ou = out + (size_t)u * kOutUnitBytes;
            float acc[E];
            // overwrite: start from writer 0; accumulate: from the owner's value
            if constexpr (ACC) {
                widen_out<OUT>(ou, acc);
            } else {
                Unit<IN>::widen(*reinterpret_cast<const uint4 *>(stage + (size_t)u * 16), acc);
            }
#pragma unroll
            for (int w = ACC ? 0 : 1; w < P; ++w) {
                float x[E];
                Unit<IN>::widen(*reinterpret_cast<const uint4 *>(stage + (size_t)w * rb + (size_t)u * 16), x);
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] = add_rn(acc[e], x[e]);
            }
            pack_out<OUT>(ou, acc);
        }
        fence_proxy_async_smem();  // the row's generic writes before the bulk store reads it
        __syncwarp();
        if (lane == 0) bulk_store((t ? p.o[1][o] : p.o[0][o]) + j * ob, out, (uint32_t)ob);
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
}

template <int P, int IN, int OUT, bool ACC>
cudaError_t launch_bulk(const GradReturnParams &p, size_t smem, cudaStream_t stream)
{
    auto kernel = grad_return_bulk_kernel<P, IN, OUT, ACC>;
    // Per device: whether the shared-memory limit is raised, and the
    // occupancy of the last shared-memory size asked for, packed into one
    // word as (smem << 8) | CTAs per SM so that concurrent callers never pair
    // one size with another's occupancy.
    static std::atomic<bool> attr_set[64];
    static std::atomic<int64_t> occupancy[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kBulkMaxSmem);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_release);
    }
    int64_t packed = occupancy[dev].load(std::memory_order_relaxed);
    if ((packed >> 8) != (int64_t)smem) {
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 32 * kBulkWarps, smem);
        if (e != cudaSuccess) return e;
        per_sm = per_sm < 1 ? 1 : (per_sm > 255 ? 255 : per_sm);
        packed = ((int64_t)smem << 8) | per_sm;
        occupancy[dev].store(packed, std::memory_order_relaxed);
    }
    int64_t blocks = (packed & 0xFF) * (int64_t)sm_count(dev);
    const int64_t needed = (p.rows + kBulkWarps - 1) / kBulkWarps;
    if (blocks > needed) blocks = needed;
    kernel<<<(unsigned)blocks, 32 * kBulkWarps, smem, stream>>>(p);
    return cudaGetLastError();
}

template <int P, int IN, int OUT, bool ACC>
cudaError_t launch_typed(const GradReturnParams &p, cudaStream_t stream)
{
    if (grad_return_uses_bulk(P, IN, OUT, ACC, p.in_row_bytes, p.rows))
        return launch_bulk<P, IN, OUT, ACC>(
            p, (size_t)kBulkWarps * ((size_t)P * p.in_row_bytes + p.out_row_bytes), stream);
    constexpr int U = P <= 4 ? 2 : 1;
    auto kernel = grad_return_kernel<P, IN, OUT, U, ACC>;
    static std::atomic<int> blocks_per_sm[64];  // per device, one table per instantiation
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

bool grad_return_uses_bulk(int P, int in_dtype, int out_dtype, bool accumulate, int64_t row_bytes,
                           int64_t rows)
{
    const int64_t out_row_bytes = row_bytes / (in_dtype == kBf16 ? 2 : 4) * (out_dtype == kBf16 ? 2 : 4);
    const int choice = g_kernel_choice.load(std::memory_order_relaxed);
    if (choice == 2) return bulk_fits(P, row_bytes, out_row_bytes);
    // One rule for both modes and for mixed types, keyed on the input rows;
    // the launch counts the output rows at their own width (twice in
    // accumulate mode, which reads them back). Measured on GB300, L2 flushed /
    // warm, against the 16-byte-load kernel:
    //  - accumulate, equal types: 0 % / +2 % at P=4 with 5 KB rows (16 GB),
    //    -9 % / -4 % at P=8, -1.5 % / +1 % at P=4 with 2 KB rows (6.7 GB),
    //    and +8 % at P=4 with 2 KB rows in a 0.8 GB launch (left to loads);
    //  - bf16 writers into float32 owners: -10 % / -6 % overwrite and
    //    -2 % / +2 % accumulate at P=4 with 5 KB rows; even at P=8; -4 % /
    //    +2 % overwrite and -5.5 % / -3 % accumulate at P=4 with 2 KB rows.
    const int64_t launch_bytes = rows * (P * row_bytes + (accumulate ? 2 : 1) * out_row_bytes);
    return choice == 0 && prefer_bulk(P, in_dtype, row_bytes, out_row_bytes, launch_bytes);
}

void set_kernel_path(int choice)
{
    g_kernel_choice.store(choice, std::memory_order_relaxed);
}

int kernel_path()
{
    return g_kernel_choice.load(std::memory_order_relaxed);
}

cudaError_t set_stall_grad_return(unsigned int extra_bytes)
{
    return cudaMemcpyToSymbol(g_stall_tx, &extra_bytes, sizeof(unsigned int));
}

cudaError_t read_wait_timeouts(unsigned int *count, bool reset)
{
    cudaError_t e = cudaMemcpyFromSymbol(count, g_wait_timeouts, sizeof(unsigned int));
    if (e == cudaSuccess && reset) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_wait_timeouts, &zero, sizeof(unsigned int));
    }
    return e;
}

cudaError_t read_grad_return_bounds_violations(unsigned int *count, bool reset)
{
    return read_bounds_counter(count, reset);
}

cudaError_t launch_grad_return(const GradReturnParams &p, int cp_size, int in_dtype,
                               int out_dtype, cudaStream_t stream, bool accumulate)
{
    if (p.rows == 0) return cudaSuccess;
    return accumulate ? launch_acc<true>(p, cp_size, in_dtype, out_dtype, stream)
                      : launch_acc<false>(p, cp_size, in_dtype, out_dtype, stream);
}

}  // namespace cpt
