// Internal launch interface between the C-ABI layer (cpt_api.cu) and the
// kernels. Not installed; callers use include/cpt.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace cpt {

constexpr int kMaxCp = 8;        // largest cp_size (one pointer slot per rank)
constexpr int kMaxTensors = 3;   // Q, K, V in one gather launch

enum Layout : int { kDualChunkSwap = 0, kPackedContiguous = 1, kDualChunkSwapPadded = 3 };
enum Dtype : int { kF32 = 0, kBf16 = 1 };

// Status codes a kernel may write to a device status word (mirror cpt.h).
constexpr int32_t kStatusTimeout = 7;
constexpr int32_t kStatusNotPublished = 10;

// Multiprocessor count of a device (queried once, cached).
int sm_count(int device);

// a1/a2: l2g[q] and, when g2l != nullptr, g2l[l2g[q]] = q for q in [0, T).
cudaError_t launch_index_map(int layout, int cp_size, const int32_t *cu, int n_docs, int64_t T,
                             int32_t *l2g, int32_t *g2l, cudaStream_t stream);

// a3: num_segs[P], seg_doc_first[P], cu_local[P][n+1], seg_offsets[P+1].
cudaError_t launch_thd_metadata(int layout, int cp_size, const int32_t *cu, int n_docs,
                                int64_t T, int32_t *num_segs, int32_t *seg_doc_first,
                                int32_t *cu_local, int32_t *seg_offsets, cudaStream_t stream);

// Padded layout maps: l2r[q] = raw row of padded local row q (-1: padding),
// r2l[g] = padded local row of raw row g.
cudaError_t launch_pad_maps(const int32_t *cu, const int32_t *cup, int n_docs, int64_t T,
                            int64_t Tpad, const int32_t *l2g_padded, const int32_t *g2l_padded,
                            int32_t *l2r, int32_t *r2l, cudaStream_t stream);

// real_len[r][i] = real tokens of document i on rank r (cup = cu if unpadded).
cudaError_t launch_real_lengths(int layout, int cp_size, const int32_t *cu, const int32_t *cup,
                                int n_docs, int64_t Tpad, int32_t *real_len, cudaStream_t stream);

// a4/a6: dst[t][r][j] = src[t][l2g[r*Tp + j]] (bit copy of 16-byte units); a
// negative index writes a zero row (padding).
struct GatherParams {
    const int32_t *l2g;                  // nullptr: identity map
    const uint8_t *src[kMaxTensors];     // [T][row_bytes]
    uint8_t *dst[kMaxTensors][kMaxCp];   // per tensor, per rank: [Tp][row_bytes]
    int64_t q0;          // first output row of the launch (flattened)
    int64_t T;           // output rows per tensor in the launch
    int64_t Tp;          // output rows per rank piece
    int64_t rows;        // n_tensors * T
    int32_t units;       // 16-byte units per row
    int32_t row_bytes;
    int64_t src_rows;    // rows of each source tensor (bounds checks)
    int32_t parts;       // destination pieces per tensor (bounds checks)
};
cudaError_t launch_gather(const GatherParams &p, cudaStream_t stream);

// a5: fused owner-gradient return for one or two tensors (dK, dV); with
// `accumulate` the owners' current values start the sums.
struct GradReturnParams {
    const int32_t *l2g;              // [T]
    const uint8_t *w[2][kMaxCp];     // writer w's global gradient [T][in_row_bytes]
    uint8_t *o[2][kMaxCp];           // owner o's local gradient [Tp][out_row_bytes]
    int64_t q0;            // first local row of the launch (flattened owner-major)
    int64_t T;             // local rows per tensor in the launch
    int64_t Tp;            // local rows per owner
    int64_t rows;          // n_tensors * T
    int32_t units;         // 16-byte input units per row
    int32_t in_row_bytes;
    int32_t out_row_bytes;
    int64_t w_rows;        // rows of each writer tensor (bounds checks)
};
// Kernel of the row gather, the fused gradient return and the slot reduce:
// 0 = the measured rule, 1 = 16-byte loads, 2 = bulk copies wherever they can
// run. Process-wide.
void set_kernel_path(int choice);
int kernel_path();

// The kernel a call runs under the current kernel path (true = the bulk-copy
// kernel). The launchers decide with these same functions.
bool gather_uses_blocks(int64_t row_bytes, int64_t rows);
bool grad_return_uses_bulk(int P, int in_dtype, int out_dtype, bool accumulate, int64_t row_bytes,
                           int64_t rows);
bool slot_reduce_uses_bulk(int P, int in_dtype, int out_dtype, int64_t bytes_per_slot);

// Reads (and, if reset, zeroes) the count of bulk-copy waits in the gradient
// return kernel that ran out of their budget, on the current device.
// Synchronous.
cudaError_t read_wait_timeouts(unsigned int *count, bool reset);
cudaError_t read_slot_reduce_wait_timeouts(unsigned int *count, bool reset);
cudaError_t read_gather_wait_timeouts(unsigned int *count, bool reset);

// Test hook: every bulk-copy mbarrier of later launches on the current device
// announces extra_bytes more than its copies deliver, so its waits run out
// (0 = normal). Synchronous.
cudaError_t set_stall_grad_return(unsigned int extra_bytes);
cudaError_t set_stall_slot_reduce(unsigned int extra_bytes);
cudaError_t set_stall_gather(unsigned int extra_bytes);

cudaError_t launch_grad_return(const GradReturnParams &p, int cp_size, int in_dtype,
                               int out_dtype, cudaStream_t stream, bool accumulate = false);

// a7: dst[i] = ordered binary32 sum of slot_0..slot_{n-1}[i].
struct SlotReduceParams {
    const uint8_t *s[kMaxCp];
    uint8_t *dst;
    int64_t n_elems;
    const int32_t *status;   // skip all work when non-null and *status != 0
};
cudaError_t launch_slot_reduce(const SlotReduceParams &p, int n_slots, int in_dtype,
                               int out_dtype, cudaStream_t stream);

// Streaming ceiling: dst = copy of srcs[0], srcs[1..n_src) read and
// discarded, through the bulk-copy engine in blocks of block_bytes and a ring
// of `stages` stages per CTA, at most ctas_per_sm CTAs per SM.
bool ceiling_shape_ok(int n_src, int block_bytes, int stages);
cudaError_t launch_stream_ceiling(const uint8_t *const *srcs, int n_src, uint8_t *dst, int64_t bytes,
                                  int block_bytes, int stages, int ctas_per_sm, cudaStream_t stream);
cudaError_t read_ceiling_wait_timeouts(unsigned int *count, bool reset);

// Failed bounds checks of each translation unit's kernels since the last
// reset (always 0 in a build without CPT_CHECK_BOUNDS). Synchronous.
cudaError_t read_index_map_bounds_violations(unsigned int *count, bool reset);
cudaError_t read_gather_bounds_violations(unsigned int *count, bool reset);
cudaError_t read_grad_return_bounds_violations(unsigned int *count, bool reset);

// Bounded epoch check: one warp polls flags_row[0..P) with acquire loads until
// every (int32)(flag - epoch) >= 0, for at most timeout_ns, then writes 0 or
// kStatusTimeout to *status.
cudaError_t launch_epoch_check(const uint32_t *flags_row, int cp_size, uint32_t epoch,
                               uint64_t timeout_ns, int32_t *status, cudaStream_t stream);

}  // namespace cpt
