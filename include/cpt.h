/*
 * cpt.h - C ABI of the context-parallel (CP) token layout and owner-gradient
 * return library for GB300 (sm_103a).
 *
 * The library models the P context-parallel ranks of one CP group as P slot
 * buffers in the HBM of ONE GPU. It computes
 *   - the two token ownership policies and their inverses,
 *   - the rank-local THD sequence metadata,
 *   - the Q/K/V reorder into rank-local order,
 *   - the fused owner-gradient return (P writers' global dK/dV summed into
 *     the owners' local gradients in binary32, writer order 0..P-1),
 *   - the staged alternative (scatter, epoch publish, bounded epoch wait,
 *     slot reduce), and the ordered one-shot sum of P slot buffers.
 *
 * Sources, by page title:
 *   [TE-3221] "[PyTorch] Add experimental packed-contiguous THD all-gather
 *             CP" (TransformerEngine PR 3221): "Why", "Scope and
 *             constraints", commit messages.
 *   [TE-3235] "Add stream-ordered CP gradient return primitive"
 *             (TransformerEngine PR 3235): "Description", "Greptile
 *             Summary", the sequence diagram, the author's reply.
 *   [NVSHMEM] "Low Latency Communication Kernels with NVSHMEM" (GPU MODE
 *             lecture 87 notes): one-shot all-reduce, exercise 3.
 *
 * Conventions that hold for every call:
 *   Memory      The caller owns every buffer. The library never allocates
 *               device memory at call time; a plan lives in a caller-provided
 *               device workspace (the only device memory of its own is the
 *               fixed array of cpt_grad_return_noalloc, part of the loaded
 *               module; the memory-management answer in "Kernel-level
 *               compute-communication overlapping for CP linear attention
 *               kernels via nvshmem", cuLA issue 15: buffers whose lifetime
 *               the caller controls; [TE-3235] "Description": peer tensor
 *               views are supplied by the caller).
 *   Pointers    "device" pointers must be device memory of the CURRENT
 *               device, 16-byte aligned. Host arrays of device pointers are
 *               read during the call only.
 *   Streams     `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *               default stream). Every call is asynchronous on it unless
 *               stated; outputs are valid once the stream reaches the call.
 *   Errors      Checks run on the host before anything is launched, and
 *               anything outside the supported scope is refused rather than
 *               attempted (as the author's reply in [TE-3235] describes its
 *               size check). On failure nothing is enqueued, the call returns a
 *               non-zero cpt_status and cpt_last_error_string() explains it.
 *               Device-side failures go to device memory the host reads:
 *               an epoch wait timeout to a status word, a bulk-copy wait
 *               that ran out to a counter (cpt_kernel_wait_timeouts), and
 *               in the bounds-checked build a failed index check to another
 *               (cpt_bounds_violations). Nothing aborts or traps.
 *   Threads     Calls are thread-safe; the error string is per thread.
 *   Graphs      cpt_index_map, cpt_thd_metadata, cpt_thd_real_lengths,
 *               cpt_partition, cpt_restore, cpt_grad_return(_accumulate),
 *               cpt_grad_scatter and cpt_slot_reduce only enqueue kernels, so
 *               they can be recorded into a CUDA graph (build the plan
 *               first). cpt_plan_create, cpt_grad_return_noalloc and the
 *               epoch publish/wait calls act on host state at call time and
 *               return CPT_ERR_UNSUPPORTED inside stream capture (as the
 *               pages' experimental CP path rejects graph capture, [TE-3221]
 *               "Scope and constraints").
 *   Layout      A "row" is the H*D elements of one token. Global tensors are
 *               [T][row]. A rank-major local tensor is [P][T/P][row]: rank
 *               r's j-th local token is flattened local index q = r*T/P + j.
 */
#ifndef CPT_H
#define CPT_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CPT_API __attribute__((visibility("default")))
#else
#define CPT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum cpt_status {
    CPT_OK = 0,
    CPT_ERR_INVALID_ARG = 1,   /* null, negative, out of range, malformed     */
    CPT_ERR_NOT_DIVISIBLE = 2, /* a partition divisibility rule fails          */
    CPT_ERR_UNSUPPORTED = 3,   /* a combination outside the validated scope    */
    CPT_ERR_ALIAS = 4,         /* outputs overlap, or the self slot mismatches */
    CPT_ERR_DEVICE = 5,        /* not device memory of the current device      */
    CPT_ERR_ALIGNMENT = 6,     /* a pointer or row size is not 16-byte aligned */
    CPT_ERR_TIMEOUT = 7,       /* (device status) epoch wait ran out of time   */
    CPT_ERR_CUDA = 8,          /* a CUDA runtime or driver call failed         */
    CPT_ERR_WORKSPACE = 9,     /* workspace too small or misaligned            */
    CPT_ERR_NOT_PUBLISHED = 10 /* wait before every writer published the epoch */
} cpt_status;

/* Token ownership policy ([TE-3221] "Why").
 *  DUAL_CHUNK_SWAP    per document: every document is cut into 2P equal
 *                     chunks; rank r owns chunks r and 2P-1-r (the owner
 *                     rule of [TE-3235], author's reply), kept in ascending
 *                     global position, documents in order. Each document length
 *                     must divide by 2P.
 *  PACKED_CONTIGUOUS  the whole packed buffer is cut into P equal contiguous
 *                     chunks, rank r owning the r-th; document boundaries
 *                     survive only through the metadata. T must divide by P.
 *  DUAL_CHUNK_SWAP_PADDED
 *                     per document, for documents of any length: each is
 *                     padded up to the next multiple of 2P (the padded
 *                     boundaries cu_padded are the prefix sums of the padded
 *                     lengths), then split as DUAL_CHUNK_SWAP over cu_padded.
 *                     This is the variant [TE-3221] "Why" contrasts with the
 *                     packed policy. T_pad = cu_padded[n] (see
 *                     cpt_plan_padded_tokens); local buffers hold T_pad/P rows
 *                     per rank, padding rows included.
 */
typedef enum cpt_layout {
    CPT_LAYOUT_DUAL_CHUNK_SWAP = 0,
    CPT_LAYOUT_PACKED_CONTIGUOUS = 1,
    CPT_LAYOUT_DUAL_CHUNK_SWAP_PADDED = 3
} cpt_layout;

/* The mirrored "packed_super_sequence" policy (2P chunks over the whole
 * packed buffer, rank r owning chunks r and 2P-1-r) was retired in favour of
 * PACKED_CONTIGUOUS as the only packed opt-in ([TE-3221] commit "Keep
 * per-document partitioning as the default ...", which keeps a negative test
 * for the retired selector). Passing this value is rejected with
 * CPT_ERR_UNSUPPORTED. Its ownership map is exactly a DUAL_CHUNK_SWAP plan
 * over cu_seqlens = {0, T}, which stays available for comparisons. */
#define CPT_LAYOUT_RETIRED_PACKED_SUPER_SEQUENCE 2

/* Element types. Sums are always accumulated in binary32. */
typedef enum cpt_dtype { CPT_F32 = 0, CPT_BF16 = 1 } cpt_dtype;

/* How cpt_epoch_wait orders the owner stream after the writers' publishes.
 *  BOUNDED  stream-ordered event waits on each writer's publish, then a
 *           one-warp kernel that re-reads the P flags with acquire loads and
 *           gives up after timeout_ns (default; can never hang).
 *  DRIVER   cuStreamWaitValue32(>= epoch) on each flag, as [TE-3235]
 *           "Description" does, then the same bounded check. The driver wait
 *           itself has no time limit, so it is only enqueued when every
 *           writer's publish of this epoch is already enqueued. */
typedef enum cpt_wait_mode { CPT_WAIT_BOUNDED = 0, CPT_WAIT_DRIVER = 1 } cpt_wait_mode;

/* Which kernel the HBM-bound calls run: the row gather, the fused gradient
 * return and the slot reduce (cpt_set_kernel_path). */
typedef enum cpt_kernel_path {
    CPT_KERNEL_AUTO = 0,  /* the measured rule (default) */
    CPT_KERNEL_LOADS = 1, /* 16-byte loads into registers */
    CPT_KERNEL_BULK = 2   /* bulk copies through shared memory, where it can run */
} cpt_kernel_path;

typedef struct cpt_plan cpt_plan;   /* opaque: layout, P, T, pointers into the workspace */
typedef struct cpt_epoch cpt_epoch; /* opaque: epoch counter and publish bookkeeping    */

/* Largest cp_size accepted. */
#define CPT_MAX_CP_SIZE 8

/* ------------------------------------------------------------------ */
/* Diagnostics                                                         */
/* ------------------------------------------------------------------ */

/* Message of the last failing call on this thread ("" if none). The pointer
 * stays valid until the next call on this thread. */
CPT_API const char *cpt_last_error_string(void);

/* Static name of a status code. */
CPT_API const char *cpt_status_string(cpt_status status);

/* ------------------------------------------------------------------ */
/* Host-only checks (no GPU needed)                                    */
/* ------------------------------------------------------------------ */

/* Validate a partition request without touching the GPU ([TE-3221] "Why"
 * and "Scope and constraints"; [TE-3235] author's reply).
 *  cu_seqlens_host  host int32[n_docs+1]: document boundaries of the packed
 *                   buffer; must start at 0, never decrease, end at
 *                   total_tokens. Zero-length documents are allowed.
 *  Returns CPT_OK; CPT_ERR_INVALID_ARG for cp_size outside 1..8, a bad
 *  layout, n_docs < 0, total_tokens outside [0, 2^31), or malformed
 *  cu_seqlens; CPT_ERR_NOT_DIVISIBLE when a document length is not a
 *  multiple of 2*cp_size (DUAL_CHUNK_SWAP) or total_tokens is not a
 *  multiple of cp_size (PACKED_CONTIGUOUS); DUAL_CHUNK_SWAP_PADDED accepts
 *  any lengths whose padded total stays below 2^31. */
CPT_API cpt_status cpt_validate_layout(cpt_layout layout, int32_t cp_size, const int32_t *cu_seqlens_host,
                               int32_t n_docs, int64_t total_tokens);

/* Device workspace bytes a plan needs (its maps and metadata), or 0 for
 * arguments that cpt_validate_layout would reject on size grounds. For
 * DUAL_CHUNK_SWAP_PADDED it is sized for the largest possible padding,
 * total_tokens + n_docs * (2*cp_size - 1). */
CPT_API size_t cpt_plan_workspace_bytes(cpt_layout layout, int32_t cp_size, int32_t n_docs,
                                int64_t total_tokens);

/* Tokens of the buffer a layout partitions, before any plan exists: for
 * DUAL_CHUNK_SWAP_PADDED every document is padded at its end to the next
 * multiple of 2*cp_size and the result is the sum of the padded lengths;
 * for the other layouts it is total_tokens. Local buffers then hold
 * padded_total/cp_size rows per rank. The pages name padding only as what
 * the packed-contiguous policy avoids ([TE-3221] "Why", "Scope and
 * constraints"); where the padding sits is this library's reading.
 *  Arguments as for cpt_validate_layout; padded_total receives the count.
 *  Host only: touches no device. The result equals cpt_plan_padded_tokens of
 *  a plan built from the same arguments.
 *  Errors: those of cpt_validate_layout (padded_total is left unchanged);
 *  CPT_ERR_INVALID_ARG for a NULL padded_total. */
CPT_API cpt_status cpt_layout_padded_tokens(cpt_layout layout, int32_t cp_size,
                                            const int32_t *cu_seqlens_host, int32_t n_docs,
                                            int64_t total_tokens, int64_t *padded_total);

/* ------------------------------------------------------------------ */
/* Plan: ownership maps and metadata, built once per batch              */
/* ------------------------------------------------------------------ */

/* Validate the request, then build the ownership maps and the metadata
 * into `workspace` on `stream` (two kernel launches and one small
 * host-to-device copy of cu_seqlens). One plan serves every later call, so
 * partition and gradient return always see the same policy ([TE-3221]
 * "Scope and constraints": partition and attention must see the same
 * selection).
 *  cu_seqlens_host  as for cpt_validate_layout; copied before the call
 *                   returns, so the caller may reuse or free it at once
 *                   (pinned host memory included).
 *  workspace        device, 256-byte aligned, >= cpt_plan_workspace_bytes;
 *                   owned by the caller, must outlive the plan and every
 *                   call that uses it.
 *  out              receives a host-side handle; free it with
 *                   cpt_plan_destroy (which does not touch the workspace).
 *  The plan is bound to the current device.
 *  Errors: those of cpt_validate_layout; CPT_ERR_WORKSPACE; CPT_ERR_DEVICE;
 *  CPT_ERR_CUDA. */
CPT_API cpt_status cpt_plan_create(cpt_layout layout, int32_t cp_size, const int32_t *cu_seqlens_host,
                           int32_t n_docs, int64_t total_tokens, void *workspace,
                           size_t workspace_bytes, void *stream, cpt_plan **out);

/* Free the host handle (NULL is accepted). Work already enqueued is not
 * affected. */
CPT_API cpt_status cpt_plan_destroy(cpt_plan *plan);

/* Total tokens T, cp_size P and document count n of a plan (any may be
 * NULL). Host only. */
CPT_API cpt_status cpt_plan_info(const cpt_plan *plan, int64_t *total_tokens, int32_t *cp_size,
                         int32_t *n_docs);

/* Tokens of the (padded) buffer the plan partitions: T_pad for
 * DUAL_CHUNK_SWAP_PADDED, T otherwise. Local buffers have T_pad/P rows per
 * rank. Host only. */
CPT_API cpt_status cpt_plan_padded_tokens(const cpt_plan *plan, int64_t *padded_total);

/* ------------------------------------------------------------------ */
/* Ownership maps                                                      */
/* ------------------------------------------------------------------ */

/* Write the local-to-global map and its inverse ([TE-3235] author's reply,
 * [TE-3221] "Why").
 *  l2g  device int32[T_pad]: l2g[q] = global token held at flattened local
 *       index q = r*T_pad/P + j (a padded position for the padded layout).
 *  g2l  device int32[T_pad] or NULL: g2l[l2g[q]] = q.
 *  DUAL_CHUNK_SWAP, document i with m = L_i/(2P) and local offset
 *  u = j - cu[i]/P inside it: l2g = cu[i] + r*m + u when u < m, else
 *  cu[i] + (2P-1-r)*m + (u-m). PACKED_CONTIGUOUS: l2g[q] = q (rank-major
 *  ownership needs no reorder, [TE-3221] commit "Allow relaxed THD
 *  all-gather ...").
 *  Errors: CPT_ERR_INVALID_ARG, CPT_ERR_DEVICE, CPT_ERR_ALIGNMENT,
 *  CPT_ERR_ALIAS (l2g and g2l overlap), CPT_ERR_CUDA. */
CPT_API cpt_status cpt_index_map(const cpt_plan *plan, int32_t *l2g, int32_t *g2l, void *stream);

/* ------------------------------------------------------------------ */
/* Rank-local THD metadata                                             */
/* ------------------------------------------------------------------ */

/* Write each rank's local sequence metadata ([TE-3221] commit "Keep
 * per-document partitioning as the default ...": one chunk and one
 * attention step per rank in packed mode, document isolation kept through
 * sequence metadata). All outputs are device int32.
 *  num_segs[P]        segments of rank r.
 *  seg_doc_first[P]   document id of rank r's first segment (-1 if none).
 *                     In packed mode a segment may start inside its
 *                     document: its keys start at global cu[doc].
 *  cu_local[P][n+1]   local segment boundaries of rank r; entries from
 *                     num_segs[r] on are T/P.
 *  seg_offsets[P+1]   exclusive prefix sum of num_segs.
 *  DUAL_CHUNK_SWAP: every rank has all n documents, cu_local = cu/P.
 *  DUAL_CHUNK_SWAP_PADDED: the same over the padded boundaries,
 *  cu_local = cu_padded/P (cpt_thd_real_lengths gives the real tokens).
 *  PACKED_CONTIGUOUS: the non-empty pieces of the documents inside
 *  [r*T/P, (r+1)*T/P), in document order, offsets relative to r*T/P.
 *  Errors: as cpt_index_map. */
CPT_API cpt_status cpt_thd_metadata(const cpt_plan *plan, int32_t *num_segs, int32_t *seg_doc_first,
                            int32_t *cu_local, int32_t *seg_offsets, void *stream);

/* Real (non-padding) tokens of every document on every rank:
 *  real_len  device int32[P][n]: real_len[r][i] = tokens of document i that
 *            rank r holds. Per-document layouts: the rank's chunks r and
 *            2P-1-r of the (padded) document, each clipped to the document's
 *            real length; packed: the document's overlap with the rank's
 *            chunk. Each column sums to the document's length.
 *  Errors: as cpt_index_map. */
CPT_API cpt_status cpt_thd_real_lengths(const cpt_plan *plan, int32_t *real_len, void *stream);

/* ------------------------------------------------------------------ */
/* Q/K/V reorder                                                       */
/* ------------------------------------------------------------------ */

/* Gather up to three token tensors into rank-local order in one launch
 * ([TE-3221] commit "Reuse the existing THD CUDA partition and reorder
 * kernels ..."): dst[t][r][j] = src[t][l2g[r*T/P + j]], a bit copy.
 *  n_tensors  1..3 (Q, K, V).
 *  src        host array of n_tensors device pointers, each [T][row].
 *  dst        host array of n_tensors device pointers, each [P][T_pad/P][row]
 *             (contiguous rank-major); must not overlap any src or another
 *             dst. Padding rows of the padded layout are written as zeros.
 *  row_elems  elements per token row (H*D); row bytes must be a multiple
 *             of 16.
 *  For PACKED_CONTIGUOUS the map is the identity: src viewed as [P][T/P][row]
 *  already is the rank-local layout (rank-major ownership requires no K/V
 *  reorder), so a caller may use that view instead; this call then performs
 *  a plain copy.
 *  Errors: CPT_ERR_INVALID_ARG, CPT_ERR_DEVICE, CPT_ERR_ALIGNMENT,
 *  CPT_ERR_ALIAS, CPT_ERR_CUDA. */
CPT_API cpt_status cpt_partition(const cpt_plan *plan, int32_t n_tensors, const void *const *src,
                         void *const *dst, int64_t row_elems, cpt_dtype dtype, void *stream);

/* cpt_partition restricted to flattened local rows [local_begin,
 * local_begin + local_count) of the rank-major output: only those rows are
 * written, each from the source row the map assigns it. Lets a caller
 * overlap host-to-device copies of one part of the batch with the reorder
 * of another. Buffers are the full tensors of cpt_partition. Errors: those
 * of cpt_partition; CPT_ERR_INVALID_ARG for a range outside [0, T_pad). */
CPT_API cpt_status cpt_partition_rows(const cpt_plan *plan, int32_t n_tensors,
                                      const void *const *src, void *const *dst, int64_t row_elems,
                                      cpt_dtype dtype, int64_t local_begin, int64_t local_count,
                                      void *stream);

/* All-gather restore: put rank-local token tensors back into global order,
 * the inverse of cpt_partition ([TE-3221] "Scope and constraints": all-gather
 * CP; commit "Allow relaxed THD all-gather ...": only rank-major ownership
 * leaves K and V in global order, so the per-document policy must reorder):
 *   dst[t][g] = src[t][g2l[g]], i.e. dst[t][l2g[q]] = src[t][q], a bit copy.
 *  src        host array of n_tensors device pointers, each [P][T_pad/P][row]
 *             (the all-gathered rank-major buffer).
 *  dst        host array of n_tensors device pointers, each [T][row] (raw
 *             order; the padded layout drops its padding rows); must not
 *             overlap any src or another dst.
 *  Other arguments and errors: as cpt_partition. */
CPT_API cpt_status cpt_restore(const cpt_plan *plan, int32_t n_tensors, const void *const *src,
                               void *const *dst, int64_t row_elems, cpt_dtype dtype, void *stream);

/* ------------------------------------------------------------------ */
/* Fused owner-gradient return                                         */
/* ------------------------------------------------------------------ */

/* Sum every writer's global dK (and dV) into each owner's local gradient
 * in one launch ([TE-3235] "Description": scatter into owner buffers in the
 * two-chunk CP layout, then accumulate the writer slots, the owner's own
 * slot included per the sequence diagram's 0..cp_size-1):
 *   out[o][j] = round(((x_0 + x_1) + x_2) + ... + x_{P-1}),
 *   x_w = (float) writer_w[l2g[o*T/P + j]],
 * binary32 adds in writer order with the accumulator starting at x_0, then
 * one rounding to the output type (round-to-nearest-even for bf16). The
 * owner buffers are overwritten.
 *  dk_writers  host array of P device pointers, writer w's global [T_pad][row]
 *              (for the padded layout: the padded global order).
 *  dk_owners   host array of P device pointers, owner o's local [T_pad/P][row].
 *  dv_writers, dv_owners  the same for dV, or both NULL to return dK only.
 *  in, out     element types of writers and owners.
 *  Errors: CPT_ERR_INVALID_ARG (one of the dV pair NULL), CPT_ERR_DEVICE,
 *  CPT_ERR_ALIGNMENT, CPT_ERR_ALIAS (an owner buffer overlaps any buffer
 *  of the call), CPT_ERR_CUDA. */
CPT_API cpt_status cpt_grad_return(const cpt_plan *plan, const void *const *dk_writers,
                           const void *const *dv_writers, void *const *dk_owners,
                           void *const *dv_owners, int64_t row_elems, cpt_dtype in,
                           cpt_dtype out, void *stream);

/* cpt_grad_return restricted to flattened owner-major local rows
 * [local_begin, local_begin + local_count): only those owner rows are
 * written, each summed from the writer rows the map assigns it, so a caller
 * can start on the rows whose writer inputs have arrived. Buffers are the
 * full tensors of cpt_grad_return. Errors: those of cpt_grad_return;
 * CPT_ERR_INVALID_ARG for a range outside [0, T_pad). */
CPT_API cpt_status cpt_grad_return_rows(const cpt_plan *plan, const void *const *dk_writers,
                                        const void *const *dv_writers, void *const *dk_owners,
                                        void *const *dv_owners, int64_t row_elems, cpt_dtype in,
                                        cpt_dtype out, int64_t local_begin, int64_t local_count,
                                        void *stream);

/* As cpt_grad_return, but the owners' current gradients start the sums (the
 * other reading of the accumulation step in [TE-3235] "Description", where
 * the owner adds its writer slots into its gradient):
 *   out[o][j] = round((((out[o][j] + x_0) + x_1) + ...) + x_{P-1}),
 * the existing owner value widened exactly to binary32 first. Each owner row
 * is read once more than in cpt_grad_return. Arguments and errors: as
 * cpt_grad_return. */
CPT_API cpt_status cpt_grad_return_accumulate(const cpt_plan *plan, const void *const *dk_writers,
                                              const void *const *dv_writers,
                                              void *const *dk_owners, void *const *dv_owners,
                                              int64_t row_elems, cpt_dtype in, cpt_dtype out,
                                              void *stream);

/* Choose the kernel of the HBM-bound calls, for the whole process and every
 * device (the pages have no counterpart: a tuning and testing control of this
 * implementation). The choice covers the row gather (cpt_partition,
 * cpt_partition_rows, cpt_restore, cpt_grad_scatter), the fused gradient
 * return (cpt_grad_return, cpt_grad_return_rows, cpt_grad_return_noalloc)
 * and cpt_slot_reduce. Both kernels of each call compute the same bits.
 *  - CPT_KERNEL_LOADS: each lane keeps 16-byte loads in flight in registers.
 *    Every case can run it.
 *  - CPT_KERNEL_BULK: data moves through shared memory with bulk copies.
 *    Row gather: blocks of up to 40 KB of consecutive rows, one bulk load
 *    per contiguous source run and one bulk store per rank piece; it needs
 *    4 blocks to fit in 200 KB. Where the map is the identity and each
 *    tensor's rank pieces lie end to end in one buffer (packed-contiguous
 *    partition and restore), the same choice runs a straight copy of 32 KB
 *    blocks instead, with no map. Gradient return: one owner row's P writer
 *    rows per warp (and, for cpt_grad_return_accumulate, the owner's current
 *    row); it needs 2 x (P x input row + output row) bytes of at most
 *    112 KB. Slot reduce: 4 KB of every slot per warp; it needs equal input
 *    and output types, and sums its last partial 4 KB with the loads
 *    kernel. Where a condition fails, the loads kernel runs.
 *  - CPT_KERNEL_AUTO (the default): bulk where it measured faster on GB300,
 *    loads elsewhere.
 *    Row gather: rows of at least 2 KB in launches that move at least
 *    384 MiB.
 *    Gradient return, either mode and any types: input rows of at least
 *    1 KB, and for P <= 6 launches of at least 2 GiB (output rows counted at
 *    their own width, twice in accumulate mode), with these input row sizes
 *    per P (by the input type):
 *      P >= 5: any row size;
 *      P = 4:  bf16 rows of at least 2 KB, float32 rows of at most 2 KB;
 *      P = 3:  bf16 rows of at least 3 KB;
 *      P <= 2: never.
 *    Slot reduce: slots of at least 1 GiB.
 *  The choice applies to calls made after this one returns. Concurrent
 *  calls from other threads see either the old or the new choice.
 *  Errors: CPT_ERR_INVALID_ARG (not one of the three values). */
CPT_API cpt_status cpt_set_kernel_path(cpt_kernel_path kernel);

/* The call families cpt_kernel_path_of answers for. */
typedef enum cpt_call {
    CPT_CALL_ROW_GATHER = 0,   /* cpt_partition(_rows), cpt_restore, cpt_grad_scatter */
    CPT_CALL_GRAD_RETURN = 1,  /* cpt_grad_return(_rows, _accumulate, _noalloc) */
    CPT_CALL_SLOT_REDUCE = 2   /* cpt_slot_reduce */
} cpt_call;

/* Which kernel a call would run under the current cpt_set_kernel_path
 * setting, with the same decision the launchers make (the pages have no
 * counterpart). Host-only; touches no device.
 *  call        the call family.
 *  cp_size     P: writers for the gradient return, slots for the slot
 *              reduce (1..8); ignored for the row gather.
 *  in, out     element types (the gather moves bytes: pass equal types).
 *  accumulate  non-zero for cpt_grad_return_accumulate.
 *  row_bytes   bytes of one row (gather, gradient return; the input row for
 *              the gradient return) or of one slot (slot reduce).
 *  rows        rows the launch writes: every tensor's rows for the gather;
 *              all owners' rows of dK (and dV) for the gradient return;
 *              ignored for the slot reduce.
 *  kernel      receives CPT_KERNEL_LOADS or CPT_KERNEL_BULK.
 *  Errors: CPT_ERR_INVALID_ARG (unknown call or type, cp_size outside
 *  1..8, a negative size, NULL kernel). */
CPT_API cpt_status cpt_kernel_path_of(cpt_call call, int32_t cp_size, cpt_dtype in, cpt_dtype out,
                                      int32_t accumulate, int64_t row_bytes, int64_t rows,
                                      cpt_kernel_path *kernel);

/* Largest batch cpt_grad_return_noalloc accepts. */
#define CPT_NOALLOC_MAX_TOKENS 1048576
#define CPT_NOALLOC_MAX_DOCS 65536

/* The fused gradient return of cpt_grad_return for callers that cannot
 * allocate device memory. Such callers include a plugin whose host
 * application owns every device byte through its own pool, and a step whose
 * memory plan is fixed before it runs. They cannot hand cpt_plan_create a
 * workspace. The pages have no counterpart to this call; it adds no
 * arithmetic, only a different home for the ownership map.
 *
 * Arguments and results are those of cpt_plan_create (layout, cp_size,
 * cu_seqlens_host, n_docs, total_tokens) followed by those of
 * cpt_grad_return; the output is bit-identical to a plan-based call. The map
 * is built into a file-scope device array inside the library instead of a
 * workspace, so the call allocates nothing:
 *  - Limits: the tokens the map covers, at most CPT_NOALLOC_MAX_TOKENS, and
 *    n_docs <= CPT_NOALLOC_MAX_DOCS. The tokens are total_tokens, except for
 *    DUAL_CHUNK_SWAP_PADDED, where they are the padded total
 *    (cpt_layout_padded_tokens), so a padded batch can be refused although
 *    its raw total is within the limit. Larger batches are rejected with
 *    CPT_ERR_INVALID_ARG and a message naming the limit. The array is
 *    (CPT_NOALLOC_MAX_DOCS + 64 + CPT_NOALLOC_MAX_TOKENS) int32, about 4.5 MB,
 *    and every GPU that loads the library holds it until the process exits.
 *  - The first call on a device looks the array's device address up with
 *    that device current (a one-time set-up that enqueues nothing); make that
 *    first call before any stream capture.
 *  - Each call uploads cu_seqlens from a host copy that lives only for the
 *    length of the call, so a call made while its stream is being captured
 *    returns CPT_ERR_UNSUPPORTED and enqueues nothing.
 *  - Every call shares the one array and leaves its map there. Calls ordered
 *    on one stream are safe; calls that overlap on the GPU (two streams, or
 *    two threads, at once) race on it and may return wrong sums.
 *  - Nothing in the array needs to start at zero: each call rewrites every
 *    map entry it reads.
 *  Errors: those of cpt_validate_layout and cpt_grad_return;
 *  CPT_ERR_UNSUPPORTED inside stream capture. */
CPT_API cpt_status cpt_grad_return_noalloc(cpt_layout layout, int32_t cp_size,
                                           const int32_t *cu_seqlens_host, int32_t n_docs,
                                           int64_t total_tokens, const void *const *dk_writers,
                                           const void *const *dv_writers, void *const *dk_owners,
                                           void *const *dv_owners, int64_t row_elems,
                                           cpt_dtype in, cpt_dtype out, void *stream);

/* ------------------------------------------------------------------ */
/* Staged owner-gradient return: scatter, publish, wait, reduce        */
/* ------------------------------------------------------------------ */

/* Scatter one writer's global gradient into its slot of every owner
 * ([TE-3235] sequence diagram: each rank copies its global dK into its slot
 * of every owner's peer_grad_key_returns): slots[o][j] = src[l2g[o*T/P + j]].
 *  writer     0..P-1.
 *  src        device [T][row].
 *  slots      host array of P device pointers: slots[o] is this writer's
 *             slot [T/P][row] in owner o's return buffer.
 *  self_slot  device pointer of the writer's own local slot as the owner
 *             sees it; must equal slots[writer] (the self-alias assertion
 *             of [TE-3235] "Greptile Summary"), else CPT_ERR_ALIAS.
 *  Errors: as cpt_partition, plus CPT_ERR_ALIAS. */
CPT_API cpt_status cpt_grad_scatter(const cpt_plan *plan, int32_t writer, const void *src,
                            void *const *slots, const void *self_slot, int64_t row_elems,
                            cpt_dtype dtype, void *stream);

/* Create the epoch state of one CP group ([TE-3235] "Description": writer
 * epochs published with cuStreamWriteValue32, waited with
 * cuStreamWaitValue32; the state is caller-owned instead of the
 * unpruned static epoch map that "Greptile Summary" flags).
 *  flags   device uint32[P][P], owner-major: flags[o*P + w] is writer w's
 *          last published epoch as seen by owner o.
 *  status  device int32[P]: status[o] is the outcome of owner o's last
 *          wait (0, CPT_ERR_TIMEOUT or CPT_ERR_NOT_PUBLISHED).
 *  Zeroes both on `stream`; the epoch counter starts at 0. Creates P CUDA
 *  events (no device memory). Errors: CPT_ERR_INVALID_ARG, CPT_ERR_DEVICE,
 *  CPT_ERR_ALIGNMENT (4-byte), CPT_ERR_ALIAS, CPT_ERR_UNSUPPORTED (driver
 *  stream memory operations unavailable), CPT_ERR_CUDA. */
CPT_API cpt_status cpt_epoch_create(int32_t cp_size, uint32_t *flags, int32_t *status, void *stream,
                            cpt_epoch **out);

/* Destroy the host state and its events. Waits for nothing. */
CPT_API cpt_status cpt_epoch_destroy(cpt_epoch *ep);

/* Start the next epoch: epoch += 1 (0 is skipped on wrap-around). Host
 * only. `epoch_out` may be NULL. */
CPT_API cpt_status cpt_epoch_advance(cpt_epoch *ep, uint32_t *epoch_out);

/* Set the current epoch to `epoch` (non-zero), e.g. to resume a saved
 * count, and forget which writers have published: every writer must
 * publish `epoch` before an owner can wait on it. Host only; the device
 * flags keep their values. Errors: CPT_ERR_INVALID_ARG for a NULL state or
 * epoch 0. */
CPT_API cpt_status cpt_epoch_set(cpt_epoch *ep, uint32_t epoch);

/* Publish the current epoch from `writer` to every owner: P driver stream
 * writes flags[o*P + writer] = epoch, each ordered after all earlier work
 * on `stream` (with the driver's default memory barrier), then an event
 * record. Errors: CPT_ERR_INVALID_ARG (writer out of range, or no epoch
 * started), CPT_ERR_DEVICE, CPT_ERR_CUDA. */
CPT_API cpt_status cpt_epoch_publish(cpt_epoch *ep, int32_t writer, void *stream);

/* Make `stream` wait until every writer has published the current epoch to
 * `owner` ([TE-3235] sequence diagram: the owner waits for every one of its
 * cp_size epoch slots to reach the epoch; here the comparison is wrap-around
 * safe, (int32)(flag - epoch) >= 0).
 *  Host check first: if some writer has not yet enqueued its publish of this
 *  epoch, nothing waits; status[owner] is set to CPT_ERR_NOT_PUBLISHED on
 *  `stream` and the call returns CPT_ERR_NOT_PUBLISHED.
 *  Otherwise `stream` is ordered after the publishes (see cpt_wait_mode),
 *  and a one-warp kernel re-reads the P flags with acquire loads, polling
 *  for at most timeout_ns (0 = a single check) and an iteration cap, then
 *  writes status[owner] = 0 or CPT_ERR_TIMEOUT. Pass `status + owner` to
 *  cpt_slot_reduce to skip the reduction after a failed wait.
 *  The writer streams must not depend on work enqueued on `stream` after
 *  this call. Errors: CPT_ERR_INVALID_ARG, CPT_ERR_NOT_PUBLISHED,
 *  CPT_ERR_DEVICE, CPT_ERR_CUDA. */
CPT_API cpt_status cpt_epoch_wait(cpt_epoch *ep, int32_t owner, uint64_t timeout_ns, cpt_wait_mode mode,
                          void *stream);

/* Synchronise `stream` and read status[owner] into *device_status.
 * Blocking, like cpt_kernel_wait_timeouts; every other call is
 * asynchronous. */
CPT_API cpt_status cpt_epoch_status(const cpt_epoch *ep, int32_t owner, void *stream,
                            int32_t *device_status);

/* Count of bounded waits inside this library's kernels that ran out of
 * their budget on the current device, since the library was loaded or last
 * reset (the pages have no counterpart: it is this implementation's failure
 * report). The bulk-copy kernels of the row gather, the gradient return and
 * the slot reduce move data through shared memory, each copy completing on
 * an mbarrier. Every wait on one gives up after about a second or 2^24 polls.
 * A wait that gives up is counted here, its warp stops, and the outputs it
 * had not reached are left unwritten. A non-zero count means some output
 * of an earlier call is not valid.
 *  count  host, receives the count.
 *  reset  non-zero: set the count back to zero after reading it.
 *  Blocking: reads device memory synchronously. Synchronise the streams of
 *  the calls you want counted first.
 *  Errors: CPT_ERR_INVALID_ARG (NULL count), CPT_ERR_DEVICE, CPT_ERR_CUDA. */
CPT_API cpt_status cpt_kernel_wait_timeouts(uint32_t *count, int32_t reset);

/* Whether this library was built with CPT_CHECK_BOUNDS (1) or not (0); the
 * pages have no counterpart. The build of context_attention_token_gb300
 * makes both: libcpt.so without the checks and libcpt_checked.so with them.
 * Host only. */
CPT_API int32_t cpt_bounds_checked(void);

/* Failed device bounds checks since the last reset (the pages have no
 * counterpart: it is this implementation's debug report). In a build with
 * CPT_CHECK_BOUNDS every index a kernel reads from memory (an ownership-map
 * entry, a document boundary) or derives from one (a rank, a local row) is
 * checked against the extent of the buffer it addresses before it is used.
 * A failed check adds one here and the access is skipped: the row is not
 * read (the gather writes it as zeros) or not written. Nothing traps. A
 * non-zero count means some earlier output is not valid. Valid inputs never
 * fail a check.
 *  count  host, receives the count.  reset  non-zero: zero it after reading.
 *  Blocking: reads device memory synchronously.
 *  Errors: CPT_ERR_UNSUPPORTED in a build without CPT_CHECK_BOUNDS;
 *  CPT_ERR_INVALID_ARG (NULL count), CPT_ERR_DEVICE, CPT_ERR_CUDA. */
CPT_API cpt_status cpt_bounds_violations(uint32_t *count, int32_t reset);

/* Test switch for the failure path of the bulk-copy kernels (the pages have no
 * counterpart). While on, every bulk-copy mbarrier of later launches on the
 * current device announces 16 bytes more than its copies deliver. Every
 * copy still completes, and nothing faults, but each wait runs out of its
 * budget (about a second). The kernels count the timeouts
 * (cpt_kernel_wait_timeouts) and stop early, leaving outputs unwritten; a
 * stalled launch takes a few seconds. Off (0) by default; turn it off
 * again before relying on any output.
 *  Blocking: writes device memory synchronously.
 *  Errors: CPT_ERR_DEVICE, CPT_ERR_CUDA. */
CPT_API cpt_status cpt_test_stall_bulk_waits(int32_t on);

/* ------------------------------------------------------------------ */
/* Ordered slot reduce                                                 */
/* ------------------------------------------------------------------ */

/* One-shot ordered sum of n_slots equally sized buffers ([TE-3235]
 * sequence diagram, where each owner sums its return slots 0..cp_size-1;
 * [NVSHMEM] one-shot all-reduce, every element reading all slots in one step):
 *   dst[i] = round(((s_0[i] + s_1[i]) + ...) + s_{n-1}[i]) in binary32.
 *  slots     host array of n_slots (1..8) device pointers, each n_elems
 *            elements of type `in`.
 *  dst       device, n_elems elements of type `out`; must not overlap a
 *            slot.
 *  status    device int32 or NULL; when non-NULL and non-zero at kernel
 *            start, the kernel writes nothing (a failed epoch wait).
 *  n_elems   any value >= 0; pointers must be 16-byte aligned.
 *  Errors: CPT_ERR_INVALID_ARG, CPT_ERR_DEVICE, CPT_ERR_ALIGNMENT,
 *  CPT_ERR_ALIAS, CPT_ERR_CUDA. */
CPT_API cpt_status cpt_slot_reduce(const void *const *slots, int32_t n_slots, int64_t n_elems,
                           cpt_dtype in, cpt_dtype out, void *dst, const int32_t *status,
                           void *stream);

/* ------------------------------------------------------------------ */
/* Measurement                                                         */
/* ------------------------------------------------------------------ */

/* Streaming ceiling for a roofline (the pages have no counterpart; it
 * computes nothing of the method). It moves the traffic of an HBM-bound call
 * with no arithmetic and no index: dst receives a copy of srcs[0], and
 * srcs[1..n_src) are read at the same offsets and discarded. With n_src = P
 * the reads and writes are those of the fused gradient return (P writer
 * rows in, one owner row out); with n_src = 1 they are those of the row
 * gather (one row in, one out). The SM's bulk-copy engine moves blocks of
 * block_bytes from every source into shared memory through a ring of
 * `stages` stages, one issuing thread per CTA and at most ctas_per_sm CTAs
 * per SM, and writes each block back with one bulk store, so the time
 * measures the memory system for that read/write mix.
 *  srcs         host array of n_src (1..8) device pointers, `bytes` each.
 *  dst          device, `bytes`; must not overlap a source.
 *  bytes        a multiple of 16 (0: nothing is launched).
 *  block_bytes  a multiple of 16; n_src * block_bytes * stages <= 200 KB.
 *  stages       2..8.  ctas_per_sm  1..32 (capped by occupancy).
 *  Bulk-copy waits that run out are counted by cpt_kernel_wait_timeouts.
 *  Errors: CPT_ERR_INVALID_ARG, CPT_ERR_ALIGNMENT, CPT_ERR_DEVICE,
 *  CPT_ERR_ALIAS, CPT_ERR_CUDA. */
CPT_API cpt_status cpt_stream_ceiling(const void *const *srcs, int32_t n_src, void *dst, int64_t bytes,
                                      int32_t block_bytes, int32_t stages, int32_t ctas_per_sm,
                                      void *stream);

#ifdef __cplusplus
}
#endif

#endif /* CPT_H */
