/*
 * Plain CPU oracle for the context-parallel (CP) token layout and the
 * owner-gradient return.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library calls this file. The
 * test suite, the smoke check and the CPU-baseline leg of the benchmark are
 * its only users. It shares no code, header or constant with the CUDA path.
 *
 * Everything here is written as obvious loops in the order the method
 * states its steps: no blocking, no fusion, no reordering. Floating point is
 * IEEE binary32 with round-to-nearest adds; build with -O2
 * -ffp-contract=off and no fast-math, so that no add is contracted or
 * reassociated.
 *
 * Sources (the pages' titles):
 *   [TE-3221] "[PyTorch] Add experimental packed-contiguous THD all-gather CP"
 *             (TransformerEngine PR 3221), commit messages and "Why".
 *   [TE-3235] "Add stream-ordered CP gradient return primitive"
 *             (TransformerEngine PR 3235), "Description", the sequence
 *             diagram, and the author's reply on CP-size genericity.
 *
 * Parity status of each function is stated in its comment.
 */
#include <stdint.h>
#include <string.h>

#define OR_LAYOUT_DSC 0    /* per-document DualChunkSwap        */
#define OR_LAYOUT_PACKED 1 /* packed-contiguous (rank-major)    */
#define OR_F32 0
#define OR_BF16 1

/* ------------------------------------------------------------------ */
/* Layout preconditions.                                               */
/* [TE-3221] "Why": the per-document partition splits every sequence   */
/* into 2*cp_size chunks, so each document length must divide by 2P;   */
/* the packed policy splits the whole buffer into cp_size equal        */
/* chunks, so T must divide by P. cu_seqlens must start at 0, never    */
/* decrease, and end at T.                                             */
/* Returns 0 if valid, 1 if malformed, 2 if a divisibility rule fails. */
/* ------------------------------------------------------------------ */
int oracle_check_layout(int layout, int P, const int32_t *cu, int n, int64_t T)
{
    if (P < 1 || n < 0 || T < 0) return 1;
    if (cu[0] != 0 || (int64_t)cu[n] != T) return 1;
    for (int i = 0; i < n; ++i)
        if (cu[i + 1] < cu[i]) return 1;
    if (layout == OR_LAYOUT_DSC) {
        for (int i = 0; i < n; ++i)
            if ((cu[i + 1] - cu[i]) % (2 * P) != 0) return 2;
    } else if (layout == OR_LAYOUT_PACKED) {
        if (T % P != 0) return 2;
    } else {
        return 1;
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Ownership of one chunk under DualChunkSwap.                         */
/* [TE-3235] author's reply: for CP size N, owner o receives native     */
/* sequence chunks o and 2N-1-o. Chunk k (0 <= k < 2N) therefore goes  */
/* to rank k when k < N and to rank 2N-1-k otherwise.                  */
/* ------------------------------------------------------------------ */
static int dsc_owner_of_chunk(int k, int P)
{
    return (k < P) ? k : (2 * P - 1 - k);
}

/* ------------------------------------------------------------------ */
/* Local-to-global token map l2g and its inverse g2l.                  */
/*                                                                     */
/* Local tokens are flattened rank-major: rank r's j-th local token is */
/* q = r*(T/P) + j.                                                    */
/*                                                                     */
/* DSC ([TE-3221] "Why", [TE-3235] reply): every document i of length  */
/* L_i is cut into 2P chunks of m_i = L_i/(2P) tokens. Rank r takes    */
/* its chunks in ascending global position, document by document       */
/* (the two-chunk CP layout named in [TE-3235] "Description").         */
/* Written as an explicit walk over every chunk of every document.     */
/*                                                                     */
/* Packed-contiguous ([TE-3221] commit "Allow relaxed THD all-gather   */
/* ..."): rank r owns the r-th of P equal contiguous pieces of the     */
/* whole buffer, so rank-major local order is global order.            */
/*                                                                     */
/* g2l may be NULL. Parity: pinned (bijection, brute force, worked     */
/* example, P=1 and packed identities).                                */
/* ------------------------------------------------------------------ */
int oracle_index_map(int layout, int P, const int32_t *cu, int n, int64_t T,
                     int32_t *l2g, int32_t *g2l)
{
    int bad = oracle_check_layout(layout, P, cu, n, T);
    if (bad) return bad;
    int64_t Tp = T / P;

    if (layout == OR_LAYOUT_DSC) {
        for (int r = 0; r < P; ++r) {
            int64_t pos = (int64_t)r * Tp;
            for (int i = 0; i < n; ++i) {
                int64_t m = (int64_t)(cu[i + 1] - cu[i]) / (2 * P);
                for (int k = 0; k < 2 * P; ++k) {
                    if (dsc_owner_of_chunk(k, P) != r) continue;
                    int64_t chunk_start = (int64_t)cu[i] + (int64_t)k * m;
                    for (int64_t t = 0; t < m; ++t) l2g[pos++] = (int32_t)(chunk_start + t);
                }
            }
        }
    } else {
        for (int r = 0; r < P; ++r)
            for (int64_t j = 0; j < Tp; ++j) l2g[(int64_t)r * Tp + j] = (int32_t)((int64_t)r * Tp + j);
    }

    if (g2l) {
        for (int64_t q = 0; q < T; ++q) g2l[l2g[q]] = (int32_t)q;
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Rank-local sequence metadata.                                       */
/*                                                                     */
/* Outputs: num_segs[P], seg_doc_first[P], cu_local[P][n+1],           */
/* seg_offsets[P+1].                                                   */
/*                                                                     */
/* DSC: every document gives each rank L_i/P tokens (two chunks), so   */
/* every rank has all n documents as segments and cu_local = cu/P.     */
/*                                                                     */
/* Packed ([TE-3221] commit "Keep per-document partitioning as the     */
/* default ...": each rank holds a single chunk and runs a single      */
/* attention step; the metadata keeps documents apart): rank r's      */
/* chunk is [a,b) = [r*T/P, (r+1)*T/P). Its segments are the non-empty */
/* intersections [cu_i, cu_{i+1}) with [a,b), in document order;       */
/* cu_local lists their starts relative to a, then b-a. Entries past   */
/* num_segs[r] repeat T/P. seg_doc_first[r] is the first document that */
/* meets the chunk (-1 when none does). Computed by plain interval     */
/* intersection.                                                       */
/*                                                                     */
/* seg_offsets is the exclusive prefix sum of num_segs.                */
/* Parity: pinned (worked example, brute-force run splitting, sums).   */
/* The packed format itself is a reading of an unspecified format.    */
/* ------------------------------------------------------------------ */
int oracle_thd_metadata(int layout, int P, const int32_t *cu, int n, int64_t T,
                        int32_t *num_segs, int32_t *seg_doc_first,
                        int32_t *cu_local, int32_t *seg_offsets)
{
    int bad = oracle_check_layout(layout, P, cu, n, T);
    if (bad) return bad;
    int64_t Tp = T / P;

    for (int r = 0; r < P; ++r) {
        int32_t *row = cu_local + (int64_t)r * (n + 1);
        if (layout == OR_LAYOUT_DSC) {
            for (int i = 0; i <= n; ++i) row[i] = cu[i] / P;
            num_segs[r] = n;
            seg_doc_first[r] = (n > 0) ? 0 : -1;
        } else {
            int64_t a = (int64_t)r * Tp, b = a + Tp;
            int k = 0, first = -1;
            for (int i = 0; i < n; ++i) {
                int64_t lo = cu[i] > a ? cu[i] : a;
                int64_t hi = cu[i + 1] < b ? cu[i + 1] : b;
                if (lo < hi) {
                    row[k++] = (int32_t)(lo - a);
                    if (first < 0) first = i;
                }
            }
            num_segs[r] = k;
            seg_doc_first[r] = first;
            for (int t = k; t <= n; ++t) row[t] = (int32_t)Tp;
        }
    }
    seg_offsets[0] = 0;
    for (int r = 0; r < P; ++r) seg_offsets[r + 1] = seg_offsets[r] + num_segs[r];
    return 0;
}

/* ------------------------------------------------------------------ */
/* Q/K/V reorder into rank-local order ([TE-3221]: "partition and      */
/* reorder kernels"): dst row q = src row l2g[q], a byte copy.         */
/* Parity: pinned (row-id payloads against the brute-force map).       */
/* ------------------------------------------------------------------ */
void oracle_partition(const int32_t *l2g, int64_t T, const void *src, void *dst,
                      int64_t row_bytes)
{
    const uint8_t *s = (const uint8_t *)src;
    uint8_t *d = (uint8_t *)dst;
    for (int64_t q = 0; q < T; ++q)
        memcpy(d + q * row_bytes, s + (int64_t)l2g[q] * row_bytes, (size_t)row_bytes);
}

/* ------------------------------------------------------------------ */
/* All-gather restore: the inverse of the reorder. After an all-gather */
/* every rank holds the rank-major buffer [P][T/P][row]; the per-      */
/* document layout must be put back into global token order before    */
/* attention sees it ([TE-3221] commit "Allow relaxed THD all-gather   */
/* ...": only rank-major ownership leaves K and V in global order).    */
/* Written as the definition: local row q goes to global row l2g[q].   */
/* Parity: pinned (round trip with the partition, brute-force map).    */
/* ------------------------------------------------------------------ */
void oracle_restore(const int32_t *l2g, int64_t T, const void *local, void *global,
                    int64_t row_bytes)
{
    const uint8_t *s = (const uint8_t *)local;
    uint8_t *d = (uint8_t *)global;
    for (int64_t q = 0; q < T; ++q)
        memcpy(d + (int64_t)l2g[q] * row_bytes, s + q * row_bytes, (size_t)row_bytes);
}

/* ------------------------------------------------------------------ */
/* Padded per-document layout: documents whose length is not a multiple */
/* of 2P ([TE-3221] "Why": the per-document partition cannot split     */
/* them) are each padded up to the next multiple of 2P. cu_padded is    */
/* the prefix sum of the padded lengths; the per-document DualChunkSwap */
/* partition then runs over cu_padded. Padding positions hold no token. */
/* Parity: pinned (divisible documents reduce to the plain layout,     */
/* round trip, zero padding rows, brute-force real-token counts).      */
/* ------------------------------------------------------------------ */
void oracle_pad_cu(int P, const int32_t *cu, int n, int32_t *cu_padded)
{
    cu_padded[0] = 0;
    for (int i = 0; i < n; ++i) {
        int32_t L = cu[i + 1] - cu[i];
        int32_t Lp = ((L + 2 * P - 1) / (2 * P)) * (2 * P);
        cu_padded[i + 1] = cu_padded[i] + Lp;
    }
}

/* Raw row held at padded global position gp, or -1 for padding. */
static int64_t raw_of_padded(const int32_t *cu, const int32_t *cup, int n, int64_t gp)
{
    for (int i = 0; i < n; ++i) {
        if (gp >= cup[i] && gp < cup[i + 1]) {
            int64_t u = gp - cup[i];
            return (u < (int64_t)(cu[i + 1] - cu[i])) ? (int64_t)cu[i] + u : -1;
        }
    }
    return -1;
}

/* Partition with padding: local row q of the padded layout receives raw row
 * raw_of_padded(l2g_padded[q]), or zero bytes for padding. Tp = Tpad/P. */
void oracle_partition_padded(const int32_t *l2g_padded, int64_t Tpad, const int32_t *cu,
                             const int32_t *cup, int n, const void *src, void *dst,
                             int64_t row_bytes)
{
    const uint8_t *s = (const uint8_t *)src;
    uint8_t *d = (uint8_t *)dst;
    for (int64_t q = 0; q < Tpad; ++q) {
        int64_t g = raw_of_padded(cu, cup, n, l2g_padded[q]);
        if (g >= 0) memcpy(d + q * row_bytes, s + g * row_bytes, (size_t)row_bytes);
        else memset(d + q * row_bytes, 0, (size_t)row_bytes);
    }
}

/* Un-pad after an all-gather: raw row g of document i sits at padded
 * position cup[i] + (g - cu[i]), which local row g2l_padded[...] holds. */
void oracle_restore_padded(const int32_t *g2l_padded, const int32_t *cu, const int32_t *cup,
                           int n, const void *local, void *raw, int64_t row_bytes)
{
    const uint8_t *s = (const uint8_t *)local;
    uint8_t *d = (uint8_t *)raw;
    for (int i = 0; i < n; ++i)
        for (int64_t g = cu[i]; g < cu[i + 1]; ++g) {
            int64_t q = g2l_padded[cup[i] + (g - cu[i])];
            memcpy(d + g * row_bytes, s + q * row_bytes, (size_t)row_bytes);
        }
}

/* Real (non-padding) tokens of document i on rank r, real_len[r*n + i], by
 * walking the rank's local rows through the map. Works for every layout:
 * pass cup = cu for the unpadded ones. */
void oracle_real_lengths(int P, const int32_t *l2g, int64_t Tpad, const int32_t *cu,
                         const int32_t *cup, int n, int32_t *real_len)
{
    int64_t Tp = Tpad / P;
    for (int64_t k = 0; k < (int64_t)P * n; ++k) real_len[k] = 0;
    for (int r = 0; r < P; ++r)
        for (int64_t j = 0; j < Tp; ++j) {
            int64_t gp = l2g[(int64_t)r * Tp + j];
            for (int i = 0; i < n; ++i)
                if (gp >= cup[i] && gp < cup[i + 1]) {
                    if (gp - cup[i] < (int64_t)(cu[i + 1] - cu[i])) real_len[r * n + i] += 1;
                    break;
                }
        }
}

/* ------------------------------------------------------------------ */
/* bf16 <-> f32.                                                       */
/* bf16 is the top half of a binary32 word, so widening is exact.      */
/* Narrowing rounds to nearest, ties to even, from the bit definition: */
/* keep the upper 16 bits, and add one when the dropped lower 16 bits  */
/* are above one half, or exactly one half with an odd kept bit. The   */
/* carry runs into the exponent, so the largest finite values round to */
/* infinity as IEEE requires. NaN inputs are outside the contract.     */
/* Parity: pinned against an independent library conversion.          */
/* ------------------------------------------------------------------ */
float oracle_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xFFFFu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

static float load_elem(const void *base, int dtype, int64_t idx)
{
    if (dtype == OR_BF16) return oracle_bf16_to_f32(((const uint16_t *)base)[idx]);
    return ((const float *)base)[idx];
}

static void store_elem(void *base, int dtype, int64_t idx, float v)
{
    if (dtype == OR_BF16)
        ((uint16_t *)base)[idx] = oracle_f32_to_bf16(v);
    else
        ((float *)base)[idx] = v;
}

/* ------------------------------------------------------------------ */
/* Ordered sum of P slot buffers ([TE-3235] sequence diagram: each     */
/* owner sums its return slots 0..cp_size-1; the one-shot sum of       */
/* "Low Latency Communication Kernels with NVSHMEM", one-shot          */
/* all-reduce). out[i] = ((s0[i] + s1[i]) + s2[i]) + ... in binary32,  */
/* the accumulator starting from slot 0 itself (so -0.0 survives),     */
/* then rounded once to the output type.                               */
/* Parity: pinned (all-ones, integer sums, order canary, -0.0, P=1,    */
/* library float32 adds).                                              */
/* ------------------------------------------------------------------ */
void oracle_slot_reduce(const void *const *slots, int P, int64_t n_elems,
                        int in_dtype, int out_dtype, void *dst)
{
    for (int64_t i = 0; i < n_elems; ++i) {
        float acc = load_elem(slots[0], in_dtype, i);
        for (int w = 1; w < P; ++w) acc = acc + load_elem(slots[w], in_dtype, i);
        store_elem(dst, out_dtype, i, acc);
    }
}

/* ------------------------------------------------------------------ */
/* Fused owner-gradient return ([TE-3235] "Description": scatter       */
/* global dK/dV into owner buffers in the two-chunk layout, then       */
/* accumulate all writer slots into the owner's gradient).             */
/*                                                                     */
/* writers[w] is writer w's global gradient [T][row]; owners[o] is     */
/* owner o's local gradient [T/P][row]. Owner o's local row j is       */
/* global row g = l2g[o*T/P + j] and receives the ordered sum over     */
/* w = 0..P-1 of writers[w][g] (the owner's own slot included: the     */
/* diagram sums every one of the cp_size slots).                       */
/* Parity: pinned through the same closed forms as slot_reduce and the */
/* map's pins.                                                         */
/* ------------------------------------------------------------------ */
void oracle_grad_return(int P, int64_t T, int64_t row_elems, int in_dtype, int out_dtype,
                        const int32_t *l2g, const void *const *writers, void *const *owners)
{
    int64_t Tp = T / P;
    for (int o = 0; o < P; ++o) {
        for (int64_t j = 0; j < Tp; ++j) {
            int64_t g = l2g[(int64_t)o * Tp + j];
            for (int64_t e = 0; e < row_elems; ++e) {
                float acc = load_elem(writers[0], in_dtype, g * row_elems + e);
                for (int w = 1; w < P; ++w)
                    acc = acc + load_elem(writers[w], in_dtype, g * row_elems + e);
                store_elem(owners[o], out_dtype, j * row_elems + e, acc);
            }
        }
    }
}

/* ------------------------------------------------------------------ */
/* Owner-gradient return that adds into the owner's existing gradient  */
/* (the other reading of the accumulation step in [TE-3235]           */
/* "Description"): the accumulator starts                              */
/* from the owner's current value, then adds writers 0..P-1 in order:  */
/*   out = round(((out + x_0) + x_1) + ... + x_{P-1}).                 */
/* Parity: pinned (ones into ones, order canary with a start value,    */
/* numpy binary32 adds).                                               */
/* ------------------------------------------------------------------ */
void oracle_grad_return_accumulate(int P, int64_t T, int64_t row_elems, int in_dtype,
                                   int out_dtype, const int32_t *l2g, const void *const *writers,
                                   void *const *owners)
{
    int64_t Tp = T / P;
    for (int o = 0; o < P; ++o) {
        for (int64_t j = 0; j < Tp; ++j) {
            int64_t g = l2g[(int64_t)o * Tp + j];
            for (int64_t e = 0; e < row_elems; ++e) {
                float acc = load_elem(owners[o], out_dtype, j * row_elems + e);
                for (int w = 0; w < P; ++w)
                    acc = acc + load_elem(writers[w], in_dtype, g * row_elems + e);
                store_elem(owners[o], out_dtype, j * row_elems + e, acc);
            }
        }
    }
}

/* ------------------------------------------------------------------ */
/* Staged scatter of one writer ([TE-3235] sequence diagram: "copy_()  */
/* scatter dk_global to peer_grad_key_returns[owner][rank]"): for      */
/* every owner o, slot row j of slots[o] = writer row l2g[o*T/P + j].  */
/* A byte copy. Parity: pinned with the partition's pins.              */
/* ------------------------------------------------------------------ */
void oracle_grad_scatter(int P, int64_t T, int64_t row_bytes, const int32_t *l2g,
                         const void *writer, void *const *slots)
{
    int64_t Tp = T / P;
    const uint8_t *s = (const uint8_t *)writer;
    for (int o = 0; o < P; ++o) {
        uint8_t *d = (uint8_t *)slots[o];
        for (int64_t j = 0; j < Tp; ++j)
            memcpy(d + j * row_bytes, s + (int64_t)l2g[(int64_t)o * Tp + j] * row_bytes,
                   (size_t)row_bytes);
    }
}
