// C ABI of the library (declared in include/cpt.h): host-side validation,
// the plan and epoch objects, and kernel dispatch.
//
// Every check runs before anything is enqueued, and unsupported input is
// refused rather than attempted ("Add stream-ordered CP gradient return
// primitive", TransformerEngine PR 3235, author's reply on its size check):
// device membership of every pointer (the page's "Greptile Summary" lists a
// current-device guard on each tensor argument), alignment, sizes, overlaps
// between outputs and every other buffer of the call, and the self-slot alias
// of the staged scatter. The driver's stream memory operations are resolved at run time
// through the runtime's driver entry-point query, so the library has no
// link-time dependency on libcuda (same page, "Changes").
#include "cpt.h"
#include "cpt_internal.h"

#include <cuda.h>
#include <nvtx3/nvToolsExt.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

namespace {

using namespace cpt;

// NVTX range named after the C-ABI call, so profilers can attribute and
// filter launches per call; without a profiler attached it costs nothing.
struct Trace {
    explicit Trace(const char *name) { nvtxRangePushA(name); }
    ~Trace() { nvtxRangePop(); }
    Trace(const Trace &) = delete;
    Trace &operator=(const Trace &) = delete;
};

thread_local std::string g_err;

cpt_status fail(cpt_status st, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return st;
}

cpt_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(CPT_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Calls whose work depends on host state at the time of the call (a plan's
// host-to-device copy of cu_seqlens, the epoch bookkeeping) cannot be
// recorded into a CUDA graph: a replay would reuse stale host decisions.
cpt_status refuse_capture(void *stream, const char *what)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cs);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return cuda_fail(e, "cudaStreamIsCapturing");
    }
    if (cs != cudaStreamCaptureStatusNone)
        return fail(CPT_ERR_UNSUPPORTED, "%s cannot be recorded into a CUDA graph: call it outside "
                    "stream capture", what);
    return CPT_OK;
}

int current_device(int *dev)
{
    return cudaGetDevice(dev) == cudaSuccess;
}

size_t dtype_size(cpt_dtype d) { return d == CPT_BF16 ? 2 : 4; }

bool dtype_ok(cpt_dtype d) { return d == CPT_F32 || d == CPT_BF16; }

// A device buffer of the current device, aligned to `align` bytes.
cpt_status check_ptr(const void *p, int device, size_t align, const char *what, int idx = -1)
{
    char name[64];
    if (idx >= 0) snprintf(name, sizeof name, "%s[%d]", what, idx);
    else snprintf(name, sizeof name, "%s", what);
    if (p == nullptr) return fail(CPT_ERR_INVALID_ARG, "%s is NULL", name);
    if (reinterpret_cast<uintptr_t>(p) % align != 0)
        return fail(CPT_ERR_ALIGNMENT, "%s is not %zu-byte aligned", name, align);
    cudaPointerAttributes a;
    cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(CPT_ERR_DEVICE, "%s is not CUDA memory (%s)", name, cudaGetErrorString(e));
    }
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)
        return fail(CPT_ERR_DEVICE, "%s is not device memory", name);
    if (a.device != device)
        return fail(CPT_ERR_DEVICE, "%s is on device %d but the current device is %d", name,
                    a.device, device);
    return CPT_OK;
}

struct Range {
    uintptr_t lo, hi;
    bool output;
    const char *what;
    int idx;
};

void add_range(std::vector<Range> &v, const void *p, size_t bytes, bool output, const char *what,
               int idx = -1)
{
    if (p == nullptr || bytes == 0) return;
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    v.push_back({lo, lo + bytes, output, what, idx});
}

// Outputs may overlap nothing; inputs may overlap each other.
cpt_status check_overlaps(const std::vector<Range> &v)
{
    for (size_t a = 0; a < v.size(); ++a)
        for (size_t b = a + 1; b < v.size(); ++b) {
            if (!v[a].output && !v[b].output) continue;
            if (v[a].lo < v[b].hi && v[b].lo < v[a].hi)
                return fail(CPT_ERR_ALIAS, "%s[%d] overlaps %s[%d]", v[a].what, v[a].idx, v[b].what,
                            v[b].idx);
        }
    return CPT_OK;
}

// ----------------------------------------------------------------- driver

typedef CUresult (*StreamValue32Fn)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);

struct DriverOps {
    StreamValue32Fn write32 = nullptr;
    StreamValue32Fn wait32 = nullptr;
    bool ok = false;
};

const DriverOps &driver_ops()
{
    static DriverOps ops;
    static std::once_flag once;
    std::call_once(once, [] {
        void *fw = nullptr, *fa = nullptr;
        cudaDriverEntryPointQueryResult qw = cudaDriverEntryPointSymbolNotFound;
        cudaDriverEntryPointQueryResult qa = cudaDriverEntryPointSymbolNotFound;
        cudaError_t ew = cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &fw, 12000,
                                                          cudaEnableDefault, &qw);
        cudaError_t ea = cudaGetDriverEntryPointByVersion("cuStreamWaitValue32", &fa, 12000,
                                                          cudaEnableDefault, &qa);
        if (ew == cudaSuccess && ea == cudaSuccess && qw == cudaDriverEntryPointSuccess &&
            qa == cudaDriverEntryPointSuccess && fw && fa) {
            ops.write32 = reinterpret_cast<StreamValue32Fn>(fw);
            ops.wait32 = reinterpret_cast<StreamValue32Fn>(fa);
            ops.ok = true;
        } else {
            cudaGetLastError();
        }
    });
    return ops;
}

// ----------------------------------------------------------------- workspace

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
    size_t cu, cup, cu_local, num_segs, first, offs, l2g, g2l, l2r, r2l, total;
};

bool is_padded(cpt_layout layout) { return layout == CPT_LAYOUT_DUAL_CHUNK_SWAP_PADDED; }

// A document of L tokens padded at its end to the next multiple of 2P.
int64_t padded_len(int64_t L, int P) { return (L + 2 * P - 1) / (2 * P) * (2 * P); }

// Sum of the padded lengths of every document.
int64_t padded_sum(const int32_t *cu, int32_t n, int P)
{
    int64_t Tpad = 0;
    for (int32_t i = 0; i < n; ++i) Tpad += padded_len((int64_t)cu[i + 1] - cu[i], P);
    return Tpad;
}

// Largest padded token count for n documents of T tokens: each document
// grows by at most 2P-1 padding tokens.
int64_t padded_cap(cpt_layout layout, int P, int n, int64_t T)
{
    return is_padded(layout) ? T + (int64_t)n * (2 * P - 1) : T;
}

WsLayout ws_layout(cpt_layout layout, int P, int n, int64_t T)
{
    const int64_t cap = padded_cap(layout, P, n, T);
    const bool pad = is_padded(layout);
    WsLayout w;
    size_t off = 0;
    w.cu = off;       off += align256(sizeof(int32_t) * (size_t)(n + 1));
    w.cup = off;      off += pad ? align256(sizeof(int32_t) * (size_t)(n + 1)) : 0;
    w.cu_local = off; off += align256(sizeof(int32_t) * (size_t)P * (size_t)(n + 1));
    w.num_segs = off; off += align256(sizeof(int32_t) * (size_t)P);
    w.first = off;    off += align256(sizeof(int32_t) * (size_t)P);
    w.offs = off;     off += align256(sizeof(int32_t) * (size_t)(P + 1));
    w.l2g = off;      off += align256(sizeof(int32_t) * (size_t)cap);
    w.g2l = off;      off += align256(sizeof(int32_t) * (size_t)cap);
    w.l2r = off;      off += pad ? align256(sizeof(int32_t) * (size_t)cap) : 0;
    w.r2l = off;      off += pad ? align256(sizeof(int32_t) * (size_t)T) : 0;
    w.total = off;
    return w;
}

cpt_status check_sizes(cpt_layout layout, int32_t P, int32_t n, int64_t T)
{
    if ((int)layout == CPT_LAYOUT_RETIRED_PACKED_SUPER_SEQUENCE)
        return fail(CPT_ERR_UNSUPPORTED,
                    "layout %d is the retired mirrored packed_super_sequence policy; use "
                    "PACKED_CONTIGUOUS, or a DUAL_CHUNK_SWAP plan over cu_seqlens = {0, T} for "
                    "its map", (int)layout);
    if (layout != CPT_LAYOUT_DUAL_CHUNK_SWAP && layout != CPT_LAYOUT_PACKED_CONTIGUOUS &&
        layout != CPT_LAYOUT_DUAL_CHUNK_SWAP_PADDED)
        return fail(CPT_ERR_INVALID_ARG, "unknown layout %d", (int)layout);
    if (P < 1 || P > CPT_MAX_CP_SIZE)
        return fail(CPT_ERR_INVALID_ARG, "cp_size %d outside 1..%d", P, CPT_MAX_CP_SIZE);
    if (n < 0 || n > 0x7FFFFFFE) return fail(CPT_ERR_INVALID_ARG, "n_docs %d out of range", n);
    if (T < 0 || T > 0x7FFFFFFF)
        return fail(CPT_ERR_INVALID_ARG, "total_tokens %lld outside [0, 2^31)", (long long)T);
    return CPT_OK;
}

}  // namespace

// ----------------------------------------------------------------- objects

struct cpt_plan {
    cpt_layout layout;
    int map_layout;   // layout the map and metadata kernels run: padded -> per-document
    int32_t P;
    int32_t n;
    int64_t T;        // tokens of the raw packed buffer
    int64_t Tpad;     // tokens after padding (= T unless padded)
    int64_t Tp;       // local tokens per rank, Tpad / P
    int device;
    const uint8_t *ws;
    size_t ws_bytes;
    int32_t *cu, *cup, *cu_local, *num_segs, *first, *offs, *l2g, *g2l, *l2r, *r2l;
    std::vector<int32_t> h_cu;   // host copy of cu_seqlens (the source of its device copy)
    std::vector<int32_t> h_cup;  // host copy of the padded boundaries
};

struct cpt_epoch {
    int32_t P;
    int device;
    uint32_t *flags;
    int32_t *status;
    uint32_t epoch;
    uint32_t published[CPT_MAX_CP_SIZE];
    cudaEvent_t ev[CPT_MAX_CP_SIZE];
    std::mutex mu;
};

namespace cpt {

int sm_count(int device)
{
    static std::mutex mu;
    static int cache[64] = {0};
    if (device < 0 && cudaGetDevice(&device) != cudaSuccess) return 1;
    if (device >= 64) return 1;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[device] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
            n <= 0)
            n = 1;
        cache[device] = n;
    }
    return cache[device];
}

}  // namespace cpt

namespace {

cpt_status check_plan(const cpt_plan *plan, int *dev)
{
    if (plan == nullptr) return fail(CPT_ERR_INVALID_ARG, "plan is NULL");
    if (!current_device(dev)) return fail(CPT_ERR_CUDA, "cudaGetDevice failed");
    if (*dev != plan->device)
        return fail(CPT_ERR_DEVICE, "plan was built on device %d but the current device is %d",
                    plan->device, *dev);
    return CPT_OK;
}

}  // namespace

extern "C" {

const char *cpt_last_error_string(void) { return g_err.c_str(); }

const char *cpt_status_string(cpt_status s)
{
    switch (s) {
    case CPT_OK: return "CPT_OK";
    case CPT_ERR_INVALID_ARG: return "CPT_ERR_INVALID_ARG";
    case CPT_ERR_NOT_DIVISIBLE: return "CPT_ERR_NOT_DIVISIBLE";
    case CPT_ERR_UNSUPPORTED: return "CPT_ERR_UNSUPPORTED";
    case CPT_ERR_ALIAS: return "CPT_ERR_ALIAS";
    case CPT_ERR_DEVICE: return "CPT_ERR_DEVICE";
    case CPT_ERR_ALIGNMENT: return "CPT_ERR_ALIGNMENT";
    case CPT_ERR_TIMEOUT: return "CPT_ERR_TIMEOUT";
    case CPT_ERR_CUDA: return "CPT_ERR_CUDA";
    case CPT_ERR_WORKSPACE: return "CPT_ERR_WORKSPACE";
    case CPT_ERR_NOT_PUBLISHED: return "CPT_ERR_NOT_PUBLISHED";
    }
    return "unknown cpt_status";
}

cpt_status cpt_validate_layout(cpt_layout layout, int32_t P, const int32_t *cu, int32_t n,
                               int64_t T)
{
    cpt_status st = check_sizes(layout, P, n, T);
    if (st) return st;
    if (cu == nullptr) return fail(CPT_ERR_INVALID_ARG, "cu_seqlens is NULL");
    if (cu[0] != 0) return fail(CPT_ERR_INVALID_ARG, "cu_seqlens[0] = %d, must be 0", cu[0]);
    if ((int64_t)cu[n] != T)
        return fail(CPT_ERR_INVALID_ARG, "cu_seqlens[%d] = %d but total_tokens = %lld", n, cu[n],
                    (long long)T);
    for (int32_t i = 0; i < n; ++i)
        if (cu[i + 1] < cu[i])
            return fail(CPT_ERR_INVALID_ARG, "cu_seqlens decreases at %d (%d -> %d)", i, cu[i],
                        cu[i + 1]);
    if (is_padded(layout)) {
        const int64_t Tpad = padded_sum(cu, n, P);
        if (Tpad > 0x7FFFFFFF)
            return fail(CPT_ERR_INVALID_ARG, "padded total %lld exceeds 2^31 - 1", (long long)Tpad);
    } else if (layout == CPT_LAYOUT_DUAL_CHUNK_SWAP) {
        for (int32_t i = 0; i < n; ++i) {
            const int32_t L = cu[i + 1] - cu[i];
            if (L % (2 * P) != 0)
                return fail(CPT_ERR_NOT_DIVISIBLE,
                            "document %d has length %d, not a multiple of 2*cp_size = %d", i, L,
                            2 * P);
        }
    } else if (T % P != 0) {
        return fail(CPT_ERR_NOT_DIVISIBLE, "total_tokens %lld is not a multiple of cp_size %d",
                    (long long)T, P);
    }
    return CPT_OK;
}

size_t cpt_plan_workspace_bytes(cpt_layout layout, int32_t P, int32_t n, int64_t T)
{
    if (check_sizes(layout, P, n, T) != CPT_OK) return 0;
    return ws_layout(layout, P, n, T).total;
}

cpt_status cpt_layout_padded_tokens(cpt_layout layout, int32_t P, const int32_t *cu, int32_t n,
                                   int64_t T, int64_t *padded_total)
{
    if (padded_total == nullptr) return fail(CPT_ERR_INVALID_ARG, "padded_total is NULL");
    cpt_status st = cpt_validate_layout(layout, P, cu, n, T);
    if (st) return st;
    *padded_total = is_padded(layout) ? padded_sum(cu, n, P) : T;
    return CPT_OK;
}

cpt_status cpt_plan_create(cpt_layout layout, int32_t P, const int32_t *cu, int32_t n, int64_t T,
                           void *workspace, size_t ws_bytes, void *stream, cpt_plan **out)
{
    Trace trace("cpt_plan_create");
    if (out == nullptr) return fail(CPT_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    cpt_status st = cpt_validate_layout(layout, P, cu, n, T);
    if (st) return st;
    int dev = 0;
    if (!current_device(&dev)) return fail(CPT_ERR_CUDA, "cudaGetDevice failed");
    if ((st = refuse_capture(stream, "cpt_plan_create"))) return st;
    const WsLayout w = ws_layout(layout, P, n, T);
    if (workspace == nullptr) return fail(CPT_ERR_WORKSPACE, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
        return fail(CPT_ERR_WORKSPACE, "workspace is not 256-byte aligned");
    if (ws_bytes < w.total)
        return fail(CPT_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, w.total);
    st = check_ptr(workspace, dev, 256, "workspace");
    if (st) return st;

    cpt_plan *p = new (std::nothrow) cpt_plan;
    if (p == nullptr) return fail(CPT_ERR_INVALID_ARG, "out of host memory");
    uint8_t *base = static_cast<uint8_t *>(workspace);
    const bool pad = is_padded(layout);
    // The device copies below read plan-owned pageable vectors, which the
    // copy stages before returning, so the caller may reuse cu_seqlens (even
    // pinned memory, whose copy would otherwise still be in flight) at once.
    try {
        p->h_cu.assign(cu, cu + (size_t)n + 1);
        if (pad) p->h_cup.resize((size_t)n + 1);
    } catch (const std::bad_alloc &) {
        delete p;
        return fail(CPT_ERR_INVALID_ARG, "out of host memory");
    }
    p->layout = layout;
    p->map_layout = pad ? (int)CPT_LAYOUT_DUAL_CHUNK_SWAP : (int)layout;
    p->P = P;
    p->n = n;
    p->T = T;
    p->device = dev;
    p->ws = base;
    p->ws_bytes = w.total;
    p->cu = reinterpret_cast<int32_t *>(base + w.cu);
    p->cu_local = reinterpret_cast<int32_t *>(base + w.cu_local);
    p->num_segs = reinterpret_cast<int32_t *>(base + w.num_segs);
    p->first = reinterpret_cast<int32_t *>(base + w.first);
    p->offs = reinterpret_cast<int32_t *>(base + w.offs);
    p->l2g = reinterpret_cast<int32_t *>(base + w.l2g);
    p->g2l = reinterpret_cast<int32_t *>(base + w.g2l);
    if (pad) {
        // every document padded up to a multiple of 2P
        p->h_cup[0] = 0;
        for (int32_t i = 0; i < n; ++i) {
            const int32_t L = cu[i + 1] - cu[i];
            p->h_cup[i + 1] = p->h_cup[i] + (int32_t)padded_len(L, P);
        }
        p->Tpad = p->h_cup[n];
        p->cup = reinterpret_cast<int32_t *>(base + w.cup);
        p->l2r = reinterpret_cast<int32_t *>(base + w.l2r);
        p->r2l = reinterpret_cast<int32_t *>(base + w.r2l);
    } else {
        p->Tpad = T;
        p->cup = p->cu;
        p->l2r = nullptr;
        p->r2l = nullptr;
    }
    p->Tp = p->Tpad / P;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(p->cu, p->h_cu.data(), sizeof(int32_t) * (size_t)(n + 1),
                                    cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess && pad)
        e = cudaMemcpyAsync(p->cup, p->h_cup.data(), sizeof(int32_t) * (size_t)(n + 1),
                            cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
        e = launch_index_map(p->map_layout, P, p->cup, n, p->Tpad, p->l2g, p->g2l, s);
    if (e == cudaSuccess && pad)
        e = launch_pad_maps(p->cu, p->cup, n, T, p->Tpad, p->l2g, p->g2l, p->l2r, p->r2l, s);
    if (e == cudaSuccess)
        e = launch_thd_metadata(p->map_layout, P, p->cup, n, p->Tpad, p->num_segs, p->first,
                                p->cu_local, p->offs, s);
    if (e != cudaSuccess) {
        delete p;
        return cuda_fail(e, "plan build");
    }
    *out = p;
    return CPT_OK;
}

cpt_status cpt_plan_destroy(cpt_plan *plan)
{
    delete plan;
    return CPT_OK;
}

cpt_status cpt_plan_info(const cpt_plan *plan, int64_t *T, int32_t *P, int32_t *n)
{
    if (plan == nullptr) return fail(CPT_ERR_INVALID_ARG, "plan is NULL");
    if (T) *T = plan->T;
    if (P) *P = plan->P;
    if (n) *n = plan->n;
    return CPT_OK;
}

cpt_status cpt_plan_padded_tokens(const cpt_plan *plan, int64_t *padded_total)
{
    if (plan == nullptr || padded_total == nullptr)
        return fail(CPT_ERR_INVALID_ARG, "NULL argument");
    *padded_total = plan->Tpad;
    return CPT_OK;
}

cpt_status cpt_index_map(const cpt_plan *plan, int32_t *l2g, int32_t *g2l, void *stream)
{
    Trace trace("cpt_index_map");
    int dev = 0;
    cpt_status st = check_plan(plan, &dev);
    if (st) return st;
    if (plan->Tpad == 0) return CPT_OK;
    if ((st = check_ptr(l2g, dev, 4, "l2g"))) return st;
    if (g2l && (st = check_ptr(g2l, dev, 4, "g2l"))) return st;
    std::vector<Range> r;
    const size_t bytes = sizeof(int32_t) * (size_t)plan->Tpad;
    add_range(r, plan->ws, plan->ws_bytes, false, "workspace");
    add_range(r, l2g, bytes, true, "l2g");
    add_range(r, g2l, bytes, true, "g2l");
    if ((st = check_overlaps(r))) return st;
    cudaError_t e = launch_index_map(plan->map_layout, plan->P, plan->cup, plan->n, plan->Tpad, l2g,
                                     g2l, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CPT_OK : cuda_fail(e, "index map launch");
}

cpt_status cpt_thd_metadata(const cpt_plan *plan, int32_t *num_segs, int32_t *seg_doc_first,
                            int32_t *cu_local, int32_t *seg_offsets, void *stream)
{
    Trace trace("cpt_thd_metadata");
    int dev = 0;
    cpt_status st = check_plan(plan, &dev);
    if (st) return st;
    if ((st = check_ptr(num_segs, dev, 4, "num_segs"))) return st;
    if ((st = check_ptr(seg_doc_first, dev, 4, "seg_doc_first"))) return st;
    if ((st = check_ptr(cu_local, dev, 4, "cu_local"))) return st;
    if ((st = check_ptr(seg_offsets, dev, 4, "seg_offsets"))) return st;
    const size_t P = (size_t)plan->P;
    std::vector<Range> r;
    add_range(r, plan->ws, plan->ws_bytes, false, "workspace");
    add_range(r, num_segs, 4 * P, true, "num_segs");
    add_range(r, seg_doc_first, 4 * P, true, "seg_doc_first");
    add_range(r, cu_local, 4 * P * (size_t)(plan->n + 1), true, "cu_local");
    add_range(r, seg_offsets, 4 * (P + 1), true, "seg_offsets");
    if ((st = check_overlaps(r))) return st;
    cudaError_t e = launch_thd_metadata(plan->map_layout, plan->P, plan->cup, plan->n, plan->Tpad,
                                        num_segs, seg_doc_first, cu_local, seg_offsets,
                                        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CPT_OK : cuda_fail(e, "metadata launch");
}

cpt_status cpt_thd_real_lengths(const cpt_plan *plan, int32_t *real_len, void *stream)
{
    Trace trace("cpt_thd_real_lengths");
    int dev = 0;
    cpt_status st = check_plan(plan, &dev);
    if (st) return st;
    const size_t count = (size_t)plan->P * (size_t)plan->n;
    if (count == 0) return CPT_OK;
    if ((st = check_ptr(real_len, dev, 4, "real_len"))) return st;
    std::vector<Range> r;
    add_range(r, plan->ws, plan->ws_bytes, false, "workspace");
    add_range(r, real_len, 4 * count, true, "real_len");
    if ((st = check_overlaps(r))) return st;
    cudaError_t e = launch_real_lengths(plan->map_layout, plan->P, plan->cu, plan->cup, plan->n,
                                        plan->Tpad, real_len, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CPT_OK : cuda_fail(e, "real lengths launch");
}

static cpt_status check_row(int64_t row_elems, cpt_dtype a, cpt_dtype b, int64_t *units)
{
    if (!dtype_ok(a) || !dtype_ok(b)) return fail(CPT_ERR_INVALID_ARG, "unknown dtype");
    if (row_elems < 1) return fail(CPT_ERR_INVALID_ARG, "row_elems %lld < 1", (long long)row_elems);
    const int64_t ra = row_elems * (int64_t)dtype_size(a), rb = row_elems * (int64_t)dtype_size(b);
    if (ra % 16 || rb % 16)
        return fail(CPT_ERR_ALIGNMENT, "row of %lld elements is not a multiple of 16 bytes",
                    (long long)row_elems);
    if (ra > (int64_t)1 << 30 || rb > (int64_t)1 << 30)
        return fail(CPT_ERR_INVALID_ARG, "row of %lld elements is too large", (long long)row_elems);
    *units = ra / 16;
    return CPT_OK;
}

// Local rows [begin, begin + count) of a plan, flattened rank-major.
static cpt_status check_local_range(const cpt_plan *plan, int64_t begin, int64_t count)
{
    if (begin < 0 || count < 0 || begin > plan->Tpad || count > plan->Tpad - begin)
        return fail(CPT_ERR_INVALID_ARG, "local rows [%lld, %lld) outside [0, %lld)",
                    (long long)begin, (long long)(begin + count), (long long)plan->Tpad);
    return CPT_OK;
}

static cpt_status partition_impl(const cpt_plan *plan, int32_t n_tensors, const void *const *src,
                                 void *const *dst, int64_t row_elems, cpt_dtype dtype,
                                 int64_t begin, int64_t count, void *stream)
{
    int dev = 0;
    cpt_status st = check_plan(plan, &dev);
    if (st) return st;
    if ((st = check_local_range(plan, begin, count))) return st;
    if (n_tensors < 1 || n_tensors > kMaxTensors)
        return fail(CPT_ERR_INVALID_ARG, "n_tensors %d outside 1..3", n_tensors);
    if (src == nullptr || dst == nullptr) return fail(CPT_ERR_INVALID_ARG, "src or dst is NULL");
    int64_t units = 0;
    if ((st = check_row(row_elems, dtype, dtype, &units))) return st;
    if (count == 0) return CPT_OK;
    const int64_t row_bytes = units * 16;
    std::vector<Range> r;
    add_range(r, plan->ws, plan->ws_bytes, false, "workspace");
    for (int t = 0; t < n_tensors; ++t) {
        if ((st = check_ptr(src[t], dev, 16, "src", t))) return st;
        if ((st = check_ptr(dst[t], dev, 16, "dst", t))) return st;
        add_range(r, src[t], (size_t)(plan->T * row_bytes), false, "src", t);
        add_range(r, dst[t], (size_t)(plan->Tpad * row_bytes), true, "dst", t);
    }
    if ((st = check_overlaps(r))) return st;

    // local row q reads raw row l2g[q] (padded layout: l2r[q], -1 = zero row)
    GatherParams p;
    memset(&p, 0, sizeof p);
    p.l2g = plan->layout == CPT_LAYOUT_PACKED_CONTIGUOUS ? nullptr
          : (is_padded(plan->layout) ? plan->l2r : plan->l2g);
    for (int t = 0; t < n_tensors; ++t) {
        p.src[t] = static_cast<const uint8_t *>(src[t]);
        for (int o = 0; o < plan->P; ++o)
            p.dst[t][o] = static_cast<uint8_t *>(dst[t]) + (int64_t)o * plan->Tp * row_bytes;
    }
    p.q0 = begin;
    p.T = count;
    p.Tp = plan->Tp;
    p.rows = (int64_t)n_tensors * count;
    p.units = (int32_t)units;
    p.row_bytes = (int32_t)row_bytes;
    p.src_rows = plan->T;
    p.parts = plan->P;
    cudaError_t e = launch_gather(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CPT_OK : cuda_fail(e, "partition launch");
}

cpt_status cpt_partition(const cpt_plan *plan, int32_t n_tensors, const void *const *src,
                         void *const *dst, int64_t row_elems, cpt_dtype dtype, void *stream)
{
    Trace trace("cpt_partition");
    if (plan == nullptr) return fail(CPT_ERR_INVALID_ARG, "plan is NULL");
    return partition_impl(plan, n_tensors, src, dst, row_elems, dtype, 0, plan->Tpad, stream);
}

cpt_status cpt_partition_rows(const cpt_plan *plan, int32_t n_tensors, const void *const *src,
                              void *const *dst, int64_t row_elems, cpt_dtype dtype,
                              int64_t local_begin, int64_t local_count, void *stream)
{
    Trace trace("cpt_partition_rows");
    return partition_impl(plan, n_tensors, src, dst, row_elems, dtype, local_begin, local_count,
                          stream);
}

cpt_status cpt_restore(const cpt_plan *plan, int32_t n_tensors, const void *const *src,
                       void *const *dst, int64_t row_elems, cpt_dtype dtype, void *stream)
{
    Trace trace("cpt_restore");
    int dev = 0;
    cpt_status st = check_plan(plan, &dev);
    if (st) return st;
    if (n_tensors < 1 || n_tensors > kMaxTensors)
        return fail(CPT_ERR_INVALID_ARG, "n_tensors %d outside 1..3", n_tensors);
    if (src == nullptr || dst == nullptr) return fail(CPT_ERR_INVALID_ARG, "src or dst is NULL");
    int64_t units = 0;
    if ((st = check_row(row_elems, dtype, dtype, &units))) return st;
    if (plan->T == 0) return CPT_OK;
    const int64_t row_bytes = units * 16;
    std::vector<Range> r;
    add_range(r, plan->ws, plan->ws_bytes, false, "workspace");
    for (int t = 0; t < n_tensors; ++t) {
        if ((st = check_ptr(src[t], dev, 16, "src", t))) return st;
        if ((st = check_ptr(dst[t], dev, 16, "dst", t))) return st;
        add_range(r, src[t], (size_t)(plan->Tpad * row_bytes), false, "src", t);
        add_range(r, dst[t], (size_t)(plan->T * row_bytes), true, "dst", t);
    }
    if ((st = check_overlaps(r))) return st;

    GatherParams p;
    memset(&p, 0, sizeof p);
    if (is_padded(plan->layout)) {
        // raw row g reads padded local row r2l[g]; the raw output is one piece
        p.l2g = plan->r2l;
        for (int t = 0; t < n_tensors; ++t) {
            p.src[t] = static_cast<const uint8_t *>(src[t]);
            p.dst[t][0] = static_cast<uint8_t *>(dst[t]);
        }
        p.Tp = plan->T;
        p.parts = 1;
    } else {
        // global row g of piece r (g = r*T/P + j) reads local row g2l[g]
        p.l2g = plan->layout == CPT_LAYOUT_PACKED_CONTIGUOUS ? nullptr : plan->g2l;
        for (int t = 0; t < n_tensors; ++t) {
            p.src[t] = static_cast<const uint8_t *>(src[t]);
            for (int o = 0; o < plan->P; ++o)
                p.dst[t][o] = static_cast<uint8_t *>(dst[t]) + (int64_t)o * plan->Tp * row_bytes;
        }
        p.Tp = plan->Tp;
        p.parts = plan->P;
    }
    p.src_rows = plan->Tpad;
    p.T = plan->T;
    p.rows = (int64_t)n_tensors * plan->T;
    p.units = (int32_t)units;
    p.row_bytes = (int32_t)row_bytes;
    cudaError_t e = launch_gather(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CPT_OK : cuda_fail(e, "restore launch");
}

static cpt_status grad_return_impl(const cpt_plan *plan, const void *const *dkw,
                                   const void *const *dvw, void *const *dko, void *const *dvo,
                                   int64_t row_elems, cpt_dtype in, cpt_dtype out, void *stream,
                                   bool accumulate, int64_t begin, int64_t count)
{
    int dev = 0;
    cpt_status st = check_plan(plan, &dev);
    if (st) return st;
    if ((st = check_local_range(plan, begin, count))) return st;
    if (dkw == nullptr || dko == nullptr)
        return fail(CPT_ERR_INVALID_ARG, "dk_writers or dk_owners is NULL");
    if ((dvw == nullptr) != (dvo == nullptr))
        return fail(CPT_ERR_INVALID_ARG, "dv_writers and dv_owners must both be given or both NULL");
    int64_t units = 0;
    if ((st = check_row(row_elems, in, out, &units))) return st;
    if (count == 0) return CPT_OK;
    const int nt = dvw ? 2 : 1;
    const int P = plan->P;
    const int64_t in_row = units * 16;
    const int64_t out_row = row_elems * (int64_t)dtype_size(out);
    const void *const *W[2] = {dkw, dvw};
    void *const *O[2] = {dko, dvo};
    static const char *wn[2] = {"dk_writers", "dv_writers"};
    static const char *on[2] = {"dk_owners", "dv_owners"};
    std::vector<Range> r;
    add_range(r, plan->ws, plan->ws_bytes, false, "workspace");
    for (int t = 0; t < nt; ++t)
        for (int w = 0; w < P; ++w) {
            if ((st = check_ptr(W[t][w], dev, 16, wn[t], w))) return st;
            if ((st = check_ptr(O[t][w], dev, 16, on[t], w))) return st;
            add_range(r, W[t][w], (size_t)(plan->Tpad * in_row), false, wn[t], w);
            add_range(r, O[t][w], (size_t)(plan->Tp * out_row), true, on[t], w);
        }
    if ((st = check_overlaps(r))) return st;

    // writers hold the (padded) global layout; owners their local rows
    GradReturnParams p;
    memset(&p, 0, sizeof p);
    p.l2g = plan->l2g;
    for (int t = 0; t < nt; ++t)
        for (int w = 0; w < P; ++w) {
            p.w[t][w] = static_cast<const uint8_t *>(W[t][w]);
            p.o[t][w] = static_cast<uint8_t *>(O[t][w]);
        }
    p.q0 = begin;
    p.T = count;
    p.Tp = plan->Tp;
    p.rows = (int64_t)nt * count;
    p.units = (int32_t)units;
    p.in_row_bytes = (int32_t)in_row;
    p.out_row_bytes = (int32_t)out_row;
    p.w_rows = plan->Tpad;
    cudaError_t e =
        launch_grad_return(p, P, in, out, static_cast<cudaStream_t>(stream), accumulate);
    return e == cudaSuccess ? CPT_OK : cuda_fail(e, "grad_return launch");
}

cpt_status cpt_grad_return(const cpt_plan *plan, const void *const *dkw, const void *const *dvw,
                           void *const *dko, void *const *dvo, int64_t row_elems, cpt_dtype in,
                           cpt_dtype out, void *stream)
{
    Trace trace("cpt_grad_return");
    if (plan == nullptr) return fail(CPT_ERR_INVALID_ARG, "plan is NULL");
    return grad_return_impl(plan, dkw, dvw, dko, dvo, row_elems, in, out, stream, false, 0,
                            plan->Tpad);
}

cpt_status cpt_grad_return_accumulate(const cpt_plan *plan, const void *const *dkw,
                                      const void *const *dvw, void *const *dko, void *const *dvo,
                                      int64_t row_elems, cpt_dtype in, cpt_dtype out, void *stream)
{
    Trace trace("cpt_grad_return_accumulate");
    if (plan == nullptr) return fail(CPT_ERR_INVALID_ARG, "plan is NULL");
    return grad_return_impl(plan, dkw, dvw, dko, dvo, row_elems, in, out, stream, true, 0,
                            plan->Tpad);
}

cpt_status cpt_grad_return_rows(const cpt_plan *plan, const void *const *dkw,
                                const void *const *dvw, void *const *dko, void *const *dvo,
                                int64_t row_elems, cpt_dtype in, cpt_dtype out, int64_t local_begin,
                                int64_t local_count, void *stream)
{
    Trace trace("cpt_grad_return_rows");
    return grad_return_impl(plan, dkw, dvw, dko, dvo, row_elems, in, out, stream, false,
                            local_begin, local_count);
}

cpt_status cpt_grad_scatter(const cpt_plan *plan, int32_t writer, const void *src,
                            void *const *slots, const void *self_slot, int64_t row_elems,
                            cpt_dtype dtype, void *stream)
{
    Trace trace("cpt_grad_scatter");
    int dev = 0;
    cpt_status st = check_plan(plan, &dev);
    if (st) return st;
    const int P = plan->P;
    if (writer < 0 || writer >= P)
        return fail(CPT_ERR_INVALID_ARG, "writer %d outside 0..%d", writer, P - 1);
    if (slots == nullptr) return fail(CPT_ERR_INVALID_ARG, "slots is NULL");
    if (slots[writer] != self_slot)
        return fail(CPT_ERR_ALIAS, "slots[%d] does not alias the writer's own local slot", writer);
    int64_t units = 0;
    if ((st = check_row(row_elems, dtype, dtype, &units))) return st;
    if (plan->Tpad == 0) return CPT_OK;
    const int64_t row_bytes = units * 16;
    std::vector<Range> r;
    add_range(r, plan->ws, plan->ws_bytes, false, "workspace");
    if ((st = check_ptr(src, dev, 16, "src"))) return st;
    add_range(r, src, (size_t)(plan->Tpad * row_bytes), false, "src");
    for (int o = 0; o < P; ++o) {
        if ((st = check_ptr(slots[o], dev, 16, "slots", o))) return st;
        add_range(r, slots[o], (size_t)(plan->Tp * row_bytes), true, "slots", o);
    }
    if ((st = check_overlaps(r))) return st;

    GatherParams p;
    memset(&p, 0, sizeof p);
    p.l2g = plan->layout == CPT_LAYOUT_PACKED_CONTIGUOUS ? nullptr : plan->l2g;
    p.src[0] = static_cast<const uint8_t *>(src);
    for (int o = 0; o < P; ++o) p.dst[0][o] = static_cast<uint8_t *>(slots[o]);
    p.T = plan->Tpad;
    p.Tp = plan->Tp;
    p.rows = plan->Tpad;
    p.units = (int32_t)units;
    p.row_bytes = (int32_t)row_bytes;
    p.src_rows = plan->Tpad;
    p.parts = P;
    cudaError_t e = launch_gather(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CPT_OK : cuda_fail(e, "grad_scatter launch");
}

cpt_status cpt_slot_reduce(const void *const *slots, int32_t n_slots, int64_t n_elems,
                           cpt_dtype in, cpt_dtype out, void *dst, const int32_t *status,
                           void *stream)
{
    Trace trace("cpt_slot_reduce");
    if (n_slots < 1 || n_slots > CPT_MAX_CP_SIZE)
        return fail(CPT_ERR_INVALID_ARG, "n_slots %d outside 1..%d", n_slots, CPT_MAX_CP_SIZE);
    if (!dtype_ok(in) || !dtype_ok(out)) return fail(CPT_ERR_INVALID_ARG, "unknown dtype");
    if (n_elems < 0) return fail(CPT_ERR_INVALID_ARG, "n_elems < 0");
    if (slots == nullptr) return fail(CPT_ERR_INVALID_ARG, "slots is NULL");
    if (n_elems == 0) return CPT_OK;
    int dev = 0;
    if (!current_device(&dev)) return fail(CPT_ERR_CUDA, "cudaGetDevice failed");
    cpt_status st;
    std::vector<Range> r;
    for (int w = 0; w < n_slots; ++w) {
        if ((st = check_ptr(slots[w], dev, 16, "slots", w))) return st;
        add_range(r, slots[w], (size_t)n_elems * dtype_size(in), false, "slots", w);
    }
    if ((st = check_ptr(dst, dev, 16, "dst"))) return st;
    add_range(r, dst, (size_t)n_elems * dtype_size(out), true, "dst");
    if (status) {
        if ((st = check_ptr(status, dev, 4, "status"))) return st;
        add_range(r, status, 4, false, "status");
    }
    if ((st = check_overlaps(r))) return st;
    SlotReduceParams p;
    memset(&p, 0, sizeof p);
    for (int w = 0; w < n_slots; ++w) p.s[w] = static_cast<const uint8_t *>(slots[w]);
    p.dst = static_cast<uint8_t *>(dst);
    p.n_elems = n_elems;
    p.status = status;
    cudaError_t e = launch_slot_reduce(p, n_slots, in, out, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CPT_OK : cuda_fail(e, "slot_reduce launch");
}

// ----------------------------------------------------------------- epochs

cpt_status cpt_epoch_create(int32_t P, uint32_t *flags, int32_t *status, void *stream,
                            cpt_epoch **out)
{
    Trace trace("cpt_epoch_create");
    if (out == nullptr) return fail(CPT_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (P < 1 || P > CPT_MAX_CP_SIZE)
        return fail(CPT_ERR_INVALID_ARG, "cp_size %d outside 1..%d", P, CPT_MAX_CP_SIZE);
    int dev = 0;
    if (!current_device(&dev)) return fail(CPT_ERR_CUDA, "cudaGetDevice failed");
    cpt_status st;
    if ((st = check_ptr(flags, dev, 4, "flags"))) return st;
    if ((st = check_ptr(status, dev, 4, "status"))) return st;
    std::vector<Range> r;
    add_range(r, flags, 4 * (size_t)P * P, true, "flags");
    add_range(r, status, 4 * (size_t)P, true, "status");
    if ((st = check_overlaps(r))) return st;
    if (!driver_ops().ok)
        return fail(CPT_ERR_UNSUPPORTED, "driver stream memory operations are unavailable");

    cpt_epoch *ep = new (std::nothrow) cpt_epoch;
    if (ep == nullptr) return fail(CPT_ERR_INVALID_ARG, "out of host memory");
    ep->P = P;
    ep->device = dev;
    ep->flags = flags;
    ep->status = status;
    ep->epoch = 0;
    for (int w = 0; w < CPT_MAX_CP_SIZE; ++w) {
        ep->published[w] = 0;
        ep->ev[w] = nullptr;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(flags, 0, 4 * (size_t)P * P, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(status, 0, 4 * (size_t)P, s);
    for (int w = 0; w < P && e == cudaSuccess; ++w)
        e = cudaEventCreateWithFlags(&ep->ev[w], cudaEventDisableTiming);
    if (e != cudaSuccess) {
        for (int w = 0; w < P; ++w)
            if (ep->ev[w]) cudaEventDestroy(ep->ev[w]);
        delete ep;
        return cuda_fail(e, "epoch create");
    }
    *out = ep;
    return CPT_OK;
}

cpt_status cpt_epoch_destroy(cpt_epoch *ep)
{
    if (ep == nullptr) return CPT_OK;
    for (int w = 0; w < ep->P; ++w)
        if (ep->ev[w]) cudaEventDestroy(ep->ev[w]);
    delete ep;
    return CPT_OK;
}

cpt_status cpt_epoch_advance(cpt_epoch *ep, uint32_t *epoch_out)
{
    if (ep == nullptr) return fail(CPT_ERR_INVALID_ARG, "epoch is NULL");
    std::lock_guard<std::mutex> lock(ep->mu);
    ep->epoch += 1;
    if (ep->epoch == 0) ep->epoch = 1;
    if (epoch_out) *epoch_out = ep->epoch;
    return CPT_OK;
}

cpt_status cpt_epoch_set(cpt_epoch *ep, uint32_t epoch)
{
    if (ep == nullptr) return fail(CPT_ERR_INVALID_ARG, "epoch is NULL");
    if (epoch == 0) return fail(CPT_ERR_INVALID_ARG, "epoch 0 is reserved for \"never published\"");
    std::lock_guard<std::mutex> lock(ep->mu);
    ep->epoch = epoch;
    for (int w = 0; w < CPT_MAX_CP_SIZE; ++w) ep->published[w] = 0;
    return CPT_OK;
}

static cpt_status check_epoch(cpt_epoch *ep, int *dev)
{
    if (ep == nullptr) return fail(CPT_ERR_INVALID_ARG, "epoch is NULL");
    if (!current_device(dev)) return fail(CPT_ERR_CUDA, "cudaGetDevice failed");
    if (*dev != ep->device)
        return fail(CPT_ERR_DEVICE, "epoch state belongs to device %d, current is %d", ep->device,
                    *dev);
    return CPT_OK;
}

cpt_status cpt_epoch_publish(cpt_epoch *ep, int32_t writer, void *stream)
{
    Trace trace("cpt_epoch_publish");
    int dev = 0;
    cpt_status st = check_epoch(ep, &dev);
    if (st) return st;
    if (writer < 0 || writer >= ep->P)
        return fail(CPT_ERR_INVALID_ARG, "writer %d outside 0..%d", writer, ep->P - 1);
    if ((st = refuse_capture(stream, "cpt_epoch_publish"))) return st;
    std::lock_guard<std::mutex> lock(ep->mu);
    if (ep->epoch == 0) return fail(CPT_ERR_INVALID_ARG, "no epoch started (call cpt_epoch_advance)");
    const DriverOps &d = driver_ops();
    CUstream s = reinterpret_cast<CUstream>(stream);
    for (int o = 0; o < ep->P; ++o) {
        CUresult r = d.write32(s, reinterpret_cast<CUdeviceptr>(ep->flags + o * ep->P + writer),
                               ep->epoch, CU_STREAM_WRITE_VALUE_DEFAULT);
        if (r != CUDA_SUCCESS) return fail(CPT_ERR_CUDA, "cuStreamWriteValue32 failed (%d)", (int)r);
    }
    cudaError_t e = cudaEventRecord(ep->ev[writer], static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "publish event record");
    ep->published[writer] = ep->epoch;
    return CPT_OK;
}

cpt_status cpt_epoch_wait(cpt_epoch *ep, int32_t owner, uint64_t timeout_ns, cpt_wait_mode mode,
                          void *stream)
{
    Trace trace("cpt_epoch_wait");
    int dev = 0;
    cpt_status st = check_epoch(ep, &dev);
    if (st) return st;
    if (owner < 0 || owner >= ep->P)
        return fail(CPT_ERR_INVALID_ARG, "owner %d outside 0..%d", owner, ep->P - 1);
    if (mode != CPT_WAIT_BOUNDED && mode != CPT_WAIT_DRIVER)
        return fail(CPT_ERR_INVALID_ARG, "unknown wait mode %d", (int)mode);
    if (timeout_ns > 10ull * 1000 * 1000 * 1000)
        return fail(CPT_ERR_INVALID_ARG, "timeout_ns above 10 s");
    if ((st = refuse_capture(stream, "cpt_epoch_wait"))) return st;
    std::lock_guard<std::mutex> lock(ep->mu);
    if (ep->epoch == 0) return fail(CPT_ERR_INVALID_ARG, "no epoch started (call cpt_epoch_advance)");
    const DriverOps &d = driver_ops();
    CUstream cs = reinterpret_cast<CUstream>(stream);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (int w = 0; w < ep->P; ++w) {
        if (ep->published[w] != ep->epoch) {
            CUresult r = d.write32(cs, reinterpret_cast<CUdeviceptr>(ep->status + owner),
                                   (cuuint32_t)kStatusNotPublished, CU_STREAM_WRITE_VALUE_DEFAULT);
            if (r != CUDA_SUCCESS)
                return fail(CPT_ERR_CUDA, "cuStreamWriteValue32 failed (%d)", (int)r);
            return fail(CPT_ERR_NOT_PUBLISHED, "writer %d has not published epoch %u", w,
                        ep->epoch);
        }
    }
    const uint32_t *row = ep->flags + owner * ep->P;
    for (int w = 0; w < ep->P; ++w) {
        if (mode == CPT_WAIT_BOUNDED) {
            cudaError_t e = cudaStreamWaitEvent(s, ep->ev[w], 0);
            if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent");
        } else {
            CUresult r = d.wait32(cs, reinterpret_cast<CUdeviceptr>(row + w), ep->epoch,
                                  CU_STREAM_WAIT_VALUE_GEQ);
            if (r != CUDA_SUCCESS)
                return fail(CPT_ERR_CUDA, "cuStreamWaitValue32 failed (%d)", (int)r);
        }
    }
    cudaError_t e = launch_epoch_check(row, ep->P, ep->epoch, timeout_ns, ep->status + owner, s);
    return e == cudaSuccess ? CPT_OK : cuda_fail(e, "epoch check launch");
}

cpt_status cpt_epoch_status(const cpt_epoch *ep, int32_t owner, void *stream, int32_t *out)
{
    Trace trace("cpt_epoch_status");
    if (ep == nullptr || out == nullptr) return fail(CPT_ERR_INVALID_ARG, "NULL argument");
    if (owner < 0 || owner >= ep->P)
        return fail(CPT_ERR_INVALID_ARG, "owner %d outside 0..%d", owner, ep->P - 1);
    int dev = 0;
    if (!current_device(&dev) || dev != ep->device)
        return fail(CPT_ERR_DEVICE, "epoch state belongs to device %d", ep->device);
    int32_t v = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(&v, ep->status + owner, 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    *out = v;
    return CPT_OK;
}

cpt_status cpt_set_kernel_path(cpt_kernel_path kernel)
{
    Trace trace("cpt_set_kernel_path");
    if (kernel != CPT_KERNEL_AUTO && kernel != CPT_KERNEL_LOADS && kernel != CPT_KERNEL_BULK)
        return fail(CPT_ERR_INVALID_ARG, "unknown kernel path %d (expected AUTO, LOADS or BULK)", (int)kernel);
    set_kernel_path((int)kernel);
    return CPT_OK;
}

cpt_status cpt_kernel_path_of(cpt_call call, int32_t cp_size, cpt_dtype in, cpt_dtype out,
                              int32_t accumulate, int64_t row_bytes, int64_t rows,
                              cpt_kernel_path *kernel)
{
    if (kernel == nullptr) return fail(CPT_ERR_INVALID_ARG, "NULL argument");
    if ((in != CPT_F32 && in != CPT_BF16) || (out != CPT_F32 && out != CPT_BF16))
        return fail(CPT_ERR_INVALID_ARG, "unknown element type");
    if (row_bytes < 0 || rows < 0) return fail(CPT_ERR_INVALID_ARG, "negative size");
    if (call != CPT_CALL_ROW_GATHER && (cp_size < 1 || cp_size > CPT_MAX_CP_SIZE))
        return fail(CPT_ERR_INVALID_ARG, "cp_size %d outside 1..%d", cp_size, CPT_MAX_CP_SIZE);
    bool bulk;
    switch (call) {
    case CPT_CALL_ROW_GATHER: bulk = gather_uses_blocks(row_bytes, rows); break;
    case CPT_CALL_GRAD_RETURN:
        bulk = grad_return_uses_bulk(cp_size, (int)in, (int)out, accumulate != 0, row_bytes, rows);
        break;
    case CPT_CALL_SLOT_REDUCE: bulk = slot_reduce_uses_bulk(cp_size, (int)in, (int)out, row_bytes); break;
    default: return fail(CPT_ERR_INVALID_ARG, "unknown call %d", (int)call);
    }
    *kernel = bulk ? CPT_KERNEL_BULK : CPT_KERNEL_LOADS;
    return CPT_OK;
}

cpt_status cpt_test_stall_bulk_waits(int32_t on)
{
    Trace trace("cpt_test_stall_bulk_waits");
    int dev = 0;
    if (!current_device(&dev)) return fail(CPT_ERR_DEVICE, "no current CUDA device");
    const unsigned int extra = on ? 16u : 0u;
    cudaError_t e = set_stall_grad_return(extra);
    if (e == cudaSuccess) e = set_stall_slot_reduce(extra);
    if (e == cudaSuccess) e = set_stall_gather(extra);
    if (e != cudaSuccess) return cuda_fail(e, "stall switch");
    return CPT_OK;
}

cpt_status cpt_kernel_wait_timeouts(uint32_t *count, int32_t reset)
{
    Trace trace("cpt_kernel_wait_timeouts");
    if (count == nullptr) return fail(CPT_ERR_INVALID_ARG, "NULL argument");
    int dev = 0;
    if (!current_device(&dev)) return fail(CPT_ERR_DEVICE, "no current CUDA device");
    unsigned int v = 0, w = 0, x = 0, y = 0;
    cudaError_t e = read_wait_timeouts(&v, reset != 0);
    if (e == cudaSuccess) e = read_slot_reduce_wait_timeouts(&w, reset != 0);
    if (e == cudaSuccess) e = read_gather_wait_timeouts(&x, reset != 0);
    if (e == cudaSuccess) e = read_ceiling_wait_timeouts(&y, reset != 0);
    if (e != cudaSuccess) return cuda_fail(e, "wait-timeout counter read");
    *count = v + w + x + y;
    return CPT_OK;
}

int32_t cpt_bounds_checked(void)
{
#ifdef CPT_CHECK_BOUNDS
    return 1;
#else
    return 0;
#endif
}

cpt_status cpt_bounds_violations(uint32_t *count, int32_t reset)
{
    Trace trace("cpt_bounds_violations");
    if (count == nullptr) return fail(CPT_ERR_INVALID_ARG, "NULL argument");
    if (!cpt_bounds_checked())
        return fail(CPT_ERR_UNSUPPORTED, "this library was built without CPT_CHECK_BOUNDS");
    int dev = 0;
    if (!current_device(&dev)) return fail(CPT_ERR_DEVICE, "no current CUDA device");
    unsigned int a = 0, b = 0, c = 0;
    cudaError_t e = read_index_map_bounds_violations(&a, reset != 0);
    if (e == cudaSuccess) e = read_gather_bounds_violations(&b, reset != 0);
    if (e == cudaSuccess) e = read_grad_return_bounds_violations(&c, reset != 0);
    if (e != cudaSuccess) return cuda_fail(e, "bounds counter read");
    *count = a + b + c;
    return CPT_OK;
}

cpt_status cpt_stream_ceiling(const void *const *srcs, int32_t n_src, void *dst, int64_t bytes,
                              int32_t block_bytes, int32_t stages, int32_t ctas_per_sm, void *stream)
{
    Trace trace("cpt_stream_ceiling");
    if (srcs == nullptr) return fail(CPT_ERR_INVALID_ARG, "srcs is NULL");
    if (!ceiling_shape_ok(n_src, block_bytes, stages))
        return fail(CPT_ERR_INVALID_ARG,
                    "n_src %d, block_bytes %d, stages %d: need 1..8 sources, 2..8 stages, blocks of "
                    "a multiple of 16 bytes and n_src * block_bytes * stages <= 200 KB",
                    n_src, block_bytes, stages);
    if (ctas_per_sm < 1 || ctas_per_sm > 32)
        return fail(CPT_ERR_INVALID_ARG, "ctas_per_sm %d outside 1..32", ctas_per_sm);
    if (bytes < 0 || bytes % 16 != 0)
        return fail(CPT_ERR_ALIGNMENT, "bytes %lld is not a non-negative multiple of 16",
                    (long long)bytes);
    int dev = 0;
    if (!current_device(&dev)) return fail(CPT_ERR_CUDA, "cudaGetDevice failed");
    if (bytes == 0) return CPT_OK;
    cpt_status st;
    std::vector<Range> r;
    const uint8_t *s8[CPT_MAX_CP_SIZE];
    for (int k = 0; k < n_src; ++k) {
        if ((st = check_ptr(srcs[k], dev, 16, "srcs", k))) return st;
        add_range(r, srcs[k], (size_t)bytes, false, "srcs", k);
        s8[k] = static_cast<const uint8_t *>(srcs[k]);
    }
    if ((st = check_ptr(dst, dev, 16, "dst"))) return st;
    add_range(r, dst, (size_t)bytes, true, "dst");
    if ((st = check_overlaps(r))) return st;
    cudaError_t e = launch_stream_ceiling(s8, n_src, static_cast<uint8_t *>(dst), bytes, block_bytes,
                                          stages, ctas_per_sm, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CPT_OK : cuda_fail(e, "stream ceiling launch");
}

}  // extern "C"

// ----------------------------------------------------------------- no allocation
//
// Fused gradient return for callers that cannot allocate device memory. Its
// map scratch is a file-scope device array, sized for at most
// CPT_NOALLOC_MAX_TOKENS tokens and CPT_NOALLOC_MAX_DOCS documents, which every
// GPU that loads this library holds until the process exits.

namespace {

constexpr int64_t kNoAllocCuSlots = CPT_NOALLOC_MAX_DOCS + 64;  // keeps the map 256-byte aligned
static __device__ __align__(256) int32_t g_noalloc_scratch[kNoAllocCuSlots + CPT_NOALLOC_MAX_TOKENS];

// Device address of g_noalloc_scratch, looked up once per device with that
// device current (host code only sees a host-side stand-in under the name).
cpt_status noalloc_scratch(int device, int32_t **out)
{
    static std::mutex mu;
    static int32_t *addr[64] = {nullptr};
    if (device < 0 || device >= 64) return fail(CPT_ERR_DEVICE, "device %d out of range", device);
    std::lock_guard<std::mutex> lock(mu);
    if (addr[device] == nullptr) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return cuda_fail(e, "cudaGetSymbolAddress of the no-allocation scratch");
        }
        addr[device] = static_cast<int32_t *>(p);
    }
    *out = addr[device];
    return CPT_OK;
}

}  // namespace

extern "C" cpt_status cpt_grad_return_noalloc(cpt_layout layout, int32_t P, const int32_t *cu,
                                              int32_t n, int64_t T, const void *const *dkw,
                                              const void *const *dvw, void *const *dko,
                                              void *const *dvo, int64_t row_elems, cpt_dtype in,
                                              cpt_dtype out, void *stream)
{
    Trace trace("cpt_grad_return_noalloc");
    cpt_status st = cpt_validate_layout(layout, P, cu, n, T);
    if (st) return st;
    // the padded layout is the per-document one over padded boundaries; the
    // other layouts copy cu_seqlens into the same vector before the upload
    std::vector<int32_t> cup;
    const int32_t *cu_map = cu;
    int64_t Tmap = T;
    int map_layout = (int)layout;
    if (is_padded(layout)) {
        try {
            cup.resize((size_t)n + 1);
        } catch (const std::bad_alloc &) {
            return fail(CPT_ERR_INVALID_ARG, "out of host memory");
        }
        cup[0] = 0;
        for (int32_t i = 0; i < n; ++i) {
            const int32_t L = cu[i + 1] - cu[i];
            cup[i + 1] = cup[i] + (int32_t)padded_len(L, P);
        }
        cu_map = cup.data();
        Tmap = cup[n];
        map_layout = (int)CPT_LAYOUT_DUAL_CHUNK_SWAP;
    }
    if (Tmap > CPT_NOALLOC_MAX_TOKENS)
        return fail(CPT_ERR_INVALID_ARG,
                    "%s %lld exceeds the no-allocation limit of %d tokens "
                    "(use cpt_plan_create with a workspace)",
                    is_padded(layout) ? "padded total" : "total_tokens", (long long)Tmap,
                    CPT_NOALLOC_MAX_TOKENS);
    if (n > CPT_NOALLOC_MAX_DOCS)
        return fail(CPT_ERR_INVALID_ARG,
                    "n_docs %d exceeds the no-allocation limit of %d documents "
                    "(use cpt_plan_create with a workspace)",
                    n, CPT_NOALLOC_MAX_DOCS);
    if (dkw == nullptr || dko == nullptr)
        return fail(CPT_ERR_INVALID_ARG, "dk_writers or dk_owners is NULL");
    if ((dvw == nullptr) != (dvo == nullptr))
        return fail(CPT_ERR_INVALID_ARG, "dv_writers and dv_owners must both be given or both NULL");
    int64_t units = 0;
    if ((st = check_row(row_elems, in, out, &units))) return st;
    int dev = 0;
    if (!current_device(&dev)) return fail(CPT_ERR_CUDA, "cudaGetDevice failed");
    // the upload below reads a host vector that dies with this call
    if ((st = refuse_capture(stream, "cpt_grad_return_noalloc"))) return st;
    int32_t *scratch = nullptr;
    if ((st = noalloc_scratch(dev, &scratch))) return st;
    if (Tmap == 0) return CPT_OK;

    const int nt = dvw ? 2 : 1;
    const int64_t Tp = Tmap / P;
    const int64_t in_row = units * 16;
    const int64_t out_row = row_elems * (int64_t)dtype_size(out);
    const void *const *W[2] = {dkw, dvw};
    void *const *O[2] = {dko, dvo};
    static const char *wn[2] = {"dk_writers", "dv_writers"};
    static const char *on[2] = {"dk_owners", "dv_owners"};
    std::vector<Range> r;
    add_range(r, scratch, sizeof(int32_t) * (size_t)(kNoAllocCuSlots + CPT_NOALLOC_MAX_TOKENS), false,
              "scratch");
    for (int t = 0; t < nt; ++t)
        for (int w = 0; w < P; ++w) {
            if ((st = check_ptr(W[t][w], dev, 16, wn[t], w))) return st;
            if ((st = check_ptr(O[t][w], dev, 16, on[t], w))) return st;
            add_range(r, W[t][w], (size_t)(Tmap * in_row), false, wn[t], w);
            add_range(r, O[t][w], (size_t)(Tp * out_row), true, on[t], w);
        }
    if ((st = check_overlaps(r))) return st;

    // every entry of the map is rewritten before it is read, so nothing in the
    // scratch has to start at zero
    int32_t *d_cu = scratch;
    int32_t *d_l2g = scratch + kNoAllocCuSlots;
    // copy from a pageable host vector, which the copy stages before
    // returning, so the caller may reuse cu_seqlens (even pinned) at once
    if (!is_padded(layout)) {
        try {
            cup.assign(cu, cu + (size_t)n + 1);
        } catch (const std::bad_alloc &) {
            return fail(CPT_ERR_INVALID_ARG, "out of host memory");
        }
        cu_map = cup.data();
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(d_cu, cu_map, sizeof(int32_t) * (size_t)(n + 1),
                                    cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = launch_index_map(map_layout, P, d_cu, n, Tmap, d_l2g, nullptr, s);
    if (e != cudaSuccess) return cuda_fail(e, "no-allocation map build");

    GradReturnParams p;
    memset(&p, 0, sizeof p);
    p.l2g = d_l2g;
    for (int t = 0; t < nt; ++t)
        for (int w = 0; w < P; ++w) {
            p.w[t][w] = static_cast<const uint8_t *>(W[t][w]);
            p.o[t][w] = static_cast<uint8_t *>(O[t][w]);
        }
    p.T = Tmap;
    p.Tp = Tp;
    p.rows = (int64_t)nt * Tmap;
    p.units = (int32_t)units;
    p.in_row_bytes = (int32_t)in_row;
    p.out_row_bytes = (int32_t)out_row;
    p.w_rows = Tmap;
    e = launch_grad_return(p, P, in, out, s);
    return e == cudaSuccess ? CPT_OK : cuda_fail(e, "grad_return launch");
}
