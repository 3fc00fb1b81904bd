// Ownership maps and rank-local THD metadata.
//
// "[PyTorch] Add experimental packed-contiguous THD all-gather CP"
// (TransformerEngine PR 3221), "Why": the per-document policy cuts every
// document into 2*cp_size chunks; the packed policy cuts the whole buffer into
// cp_size equal chunks. "Add stream-ordered CP gradient return primitive"
// (TransformerEngine PR 3235), author's reply: owner o receives chunks o and
// 2N-1-o.
//
// The kernels here (the map, the metadata, the padded layout's extra maps
// and the real-token counts) are integer-only and move a few bytes per token;
// they are launch-bound at the sizes used here, so they favour simplicity.
#include "cpt_device.cuh"
#include "cpt_internal.h"

namespace cpt {

namespace {

// Closed form of the DualChunkSwap map for flattened local index q: find the
// document whose local range [cu[i]/P, cu[i+1]/P) holds j, then place j in
// the rank's early chunk (r) or late chunk (2P-1-r) of that document.
__global__ void index_map_kernel(int layout, int P, const int32_t *__restrict__ cu, int n,
                                 int64_t T, int32_t *__restrict__ l2g,
                                 int32_t *__restrict__ g2l)
{
    const int64_t Tp = T / P;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < T; q += stride) {
        int64_t g;
        if (layout == kDualChunkSwap) {
            const int64_t r = q / Tp;
            const int64_t j = q - r * Tp;
            // last i in [0, n) with cu[i]/P <= j (zero-length documents share
            // a start and are skipped because the next start is larger)
            int lo = 0, hi = n;  // invariant: cu[lo]/P <= j < cu[hi]/P
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (__ldg(cu + mid) / P <= j) lo = mid; else hi = mid;
            }
            if constexpr (kCheckBounds) {
                if (!in_bounds(lo >= 0 && lo < n)) continue;
            }
            const int64_t c0 = __ldg(cu + lo);
            const int64_t m = (__ldg(cu + lo + 1) - c0) / (2 * P);
            const int64_t u = j - c0 / P;
            g = (u < m) ? c0 + r * m + u : c0 + (2 * P - 1 - r) * m + (u - m);
        } else {
            g = q;
        }
        if constexpr (kCheckBounds) {
            if (!in_bounds(g >= 0 && g < T)) continue;
        }
        l2g[q] = (int32_t)g;
        if (g2l) g2l[g] = (int32_t)q;
    }
}

// One CTA; warp r builds rank r's metadata. Packed mode compacts the
// non-empty document pieces with a warp ballot; warp 0 then scans the counts.
__global__ void thd_metadata_kernel(int layout, int P, const int32_t *__restrict__ cu, int n,
                                    int64_t T, int32_t *__restrict__ num_segs,
                                    int32_t *__restrict__ seg_doc_first,
                                    int32_t *__restrict__ cu_local,
                                    int32_t *__restrict__ seg_offsets)
{
    __shared__ int32_t s_count[kMaxCp];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t Tp = T / P;

    if (warp < P) {
        const int r = warp;
        int32_t *row = cu_local + (int64_t)r * (n + 1);
        if (layout == kDualChunkSwap) {
            for (int i = lane; i <= n; i += 32) row[i] = __ldg(cu + i) / P;
            if (lane == 0) {
                num_segs[r] = n;
                seg_doc_first[r] = n > 0 ? 0 : -1;
                s_count[r] = n;
            }
        } else {
            const int64_t a = (int64_t)r * Tp, b = a + Tp;
            int count = 0, first = -1;
            for (int base = 0; base < n; base += 32) {
                const int i = base + lane;
                int64_t lo = 0;
                bool nonempty = false;
                if (i < n) {
                    const int64_t c0 = __ldg(cu + i), c1 = __ldg(cu + i + 1);
                    lo = c0 > a ? c0 : a;
                    const int64_t hi = c1 < b ? c1 : b;
                    nonempty = lo < hi;
                }
                const unsigned ballot = __ballot_sync(0xFFFFFFFFu, nonempty);
                const int slot = count + __popc(ballot & ((1u << lane) - 1u));
                if (nonempty && in_bounds(slot <= n)) row[slot] = (int32_t)(lo - a);
                if (first < 0 && ballot) first = base + __ffs(ballot) - 1;
                count += __popc(ballot);
            }
            for (int t = count + lane; t <= n; t += 32) row[t] = (int32_t)Tp;
            if (lane == 0) {
                num_segs[r] = count;
                seg_doc_first[r] = first;
                s_count[r] = count;
            }
        }
    }
    __syncthreads();
    if (warp == 0) {
        int v = lane < P ? s_count[lane] : 0;
        int incl = v;
        for (int d = 1; d < 32; d <<= 1) {
            const int up = __shfl_up_sync(0xFFFFFFFFu, incl, d);
            if (lane >= d) incl += up;
        }
        if (lane == 0) seg_offsets[0] = 0;
        if (lane < P) seg_offsets[lane + 1] = incl;
    }
}

// Padded per-document layout: documents are padded up to multiples of 2P
// (cup = padded prefix sums). l2r[q]: raw row held by padded local row q, or
// -1 for padding; r2l[g]: padded local row holding raw row g.
__global__ void pad_maps_kernel(const int32_t *__restrict__ cu, const int32_t *__restrict__ cup,
                                int n, int64_t T, int64_t Tpad,
                                const int32_t *__restrict__ l2g_padded,
                                const int32_t *__restrict__ g2l_padded, int32_t *__restrict__ l2r,
                                int32_t *__restrict__ r2l)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < Tpad; q += stride) {
        const int64_t gp = __ldg(l2g_padded + q);
        int lo = 0, hi = n;  // last i with cup[i] <= gp (gp < cup[n] = Tpad)
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(cup + mid) <= gp) lo = mid; else hi = mid;
        }
        if constexpr (kCheckBounds) {
            if (!in_bounds(gp >= 0 && gp < Tpad && lo >= 0 && lo < n)) continue;
        }
        const int64_t u = gp - __ldg(cup + lo);
        const int64_t L = __ldg(cu + lo + 1) - __ldg(cu + lo);
        l2r[q] = u < L ? (int32_t)(__ldg(cu + lo) + u) : -1;
    }
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < T; g += stride) {
        int lo = 0, hi = n;  // last i with cu[i] <= g (g < cu[n] = T)
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(cu + mid) <= g) lo = mid; else hi = mid;
        }
        const int64_t gp = __ldg(cup + lo) + (g - __ldg(cu + lo));
        if constexpr (kCheckBounds) {
            if (!in_bounds(lo >= 0 && lo < n && gp >= 0 && gp < Tpad)) continue;
        }
        r2l[g] = __ldg(g2l_padded + gp);
    }
}

// real_len[r][i]: real tokens of document i on rank r. Per-document layouts
// (cup = cu when unpadded): the rank's chunks r and 2P-1-r of the padded
// document, each clipped to the real length. Packed: the document's overlap
// with the rank's contiguous chunk.
__global__ void real_lengths_kernel(int layout, int P, const int32_t *__restrict__ cu,
                                    const int32_t *__restrict__ cup, int n, int64_t Tpad,
                                    int32_t *__restrict__ real_len)
{
    const int64_t total = (int64_t)P * n;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < total; k += stride) {
        const int r = (int)(k / n);
        const int i = (int)(k - (int64_t)r * n);
        const int64_t c0 = __ldg(cu + i), L = __ldg(cu + i + 1) - c0;
        int64_t v = 0;
        if (layout == kPackedContiguous) {
            const int64_t Tp = Tpad / P, a = (int64_t)r * Tp, b = a + Tp;
            const int64_t lo = c0 > a ? c0 : a, hi = c0 + L < b ? c0 + L : b;
            v = hi > lo ? hi - lo : 0;
        } else {
            const int64_t mp = (__ldg(cup + i + 1) - __ldg(cup + i)) / (2 * P);
            const int64_t ks[2] = {r, 2 * P - 1 - r};
            for (int h = 0; h < 2; ++h) {
                int64_t c = L - ks[h] * mp;
                c = c < 0 ? 0 : (c > mp ? mp : c);
                v += c;
            }
        }
        real_len[k] = (int32_t)v;
    }
}

}  // namespace

cudaError_t read_index_map_bounds_violations(unsigned int *count, bool reset)
{
    return read_bounds_counter(count, reset);
}

cudaError_t launch_index_map(int layout, int cp_size, const int32_t *cu, int n_docs, int64_t T,
                             int32_t *l2g, int32_t *g2l, cudaStream_t stream)
{
    if (T == 0) return cudaSuccess;
    const int threads = 256;
    int64_t blocks = (T + threads - 1) / threads;
    const int64_t cap = (int64_t)sm_count(-1) * 8;
    if (blocks > cap) blocks = cap;
    index_map_kernel<<<(unsigned)blocks, threads, 0, stream>>>(layout, cp_size, cu, n_docs, T,
                                                                l2g, g2l);
    return cudaGetLastError();
}

cudaError_t launch_thd_metadata(int layout, int cp_size, const int32_t *cu, int n_docs,
                                int64_t T, int32_t *num_segs, int32_t *seg_doc_first,
                                int32_t *cu_local, int32_t *seg_offsets, cudaStream_t stream)
{
    thd_metadata_kernel<<<1, 32 * kMaxCp, 0, stream>>>(layout, cp_size, cu, n_docs, T, num_segs,
                                                        seg_doc_first, cu_local, seg_offsets);
    return cudaGetLastError();
}

}  // namespace cpt

namespace cpt {

cudaError_t launch_pad_maps(const int32_t *cu, const int32_t *cup, int n_docs, int64_t T,
                            int64_t Tpad, const int32_t *l2g_padded, const int32_t *g2l_padded,
                            int32_t *l2r, int32_t *r2l, cudaStream_t stream)
{
    const int64_t work = Tpad > T ? Tpad : T;
    if (work == 0) return cudaSuccess;
    const int threads = 256;
    int64_t blocks = (work + threads - 1) / threads;
    const int64_t cap = (int64_t)sm_count(-1) * 8;
    if (blocks > cap) blocks = cap;
    pad_maps_kernel<<<(unsigned)blocks, threads, 0, stream>>>(cu, cup, n_docs, T, Tpad, l2g_padded,
                                                              g2l_padded, l2r, r2l);
    return cudaGetLastError();
}

cudaError_t launch_real_lengths(int layout, int cp_size, const int32_t *cu, const int32_t *cup,
                                int n_docs, int64_t Tpad, int32_t *real_len, cudaStream_t stream)
{
    const int64_t total = (int64_t)cp_size * n_docs;
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    if (blocks > 1024) blocks = 1024;
    real_lengths_kernel<<<(unsigned)blocks, threads, 0, stream>>>(layout, cp_size, cu, cup, n_docs,
                                                                  Tpad, real_len);
    return cudaGetLastError();
}

}  // namespace cpt
