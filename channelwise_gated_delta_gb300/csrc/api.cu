// api.cu -- the C ABI declared in include/gdr.h: argument validation,
// routing by sequence length (page "Reorder channelwise gated delta rule
// chunked hot loops for autovectorization", pytorch/executorch PR #21021,
// second commit summary: T == 1 runs the two-pass token recurrence, T != 1
// the chunkwise WY/UT form), workspace management and launches.
#include <algorithm>
#include <mutex>
#include <stdint.h>
#include <string.h>
#include <vector>

#include "common.cuh"
#include "gdr.h"

// Device-wide error word: kernels that wait with a bounded spin set it
// instead of hanging; gdr_device_check reads and clears it.
__device__ int g_gdr_device_error = 0;

namespace {

thread_local int t_last_cuda_error = 0;

gdr_status cuda_fail(cudaError_t e) {
    t_last_cuda_error = (int)e;
    return GDR_ERR_CUDA;
}

bool supported_dim(int d) { return d == 32 || d == 64 || d == 128; }
bool supported_chunk(int c) { return c == 16 || c == 32 || c == 64; }
bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};
Range range_of(const void *p, size_t bytes) {
    return Range{(uintptr_t)p, (uintptr_t)p + bytes};
}
bool overlap(Range a, Range b) {
    return a.lo != a.hi && b.lo != b.hi && a.lo < b.hi && b.lo < a.hi;
}

// Validates pointers for BT token rows and NS state slots (alignment,
// overlap); the shape checks common to every entry point.
gdr_status validate_rows(const void *q, const void *k, const void *v, const float *g,
                         const float *beta, const float *h0, void *out, float *ht, long long BT,
                         long long NS, int HK, int HV, int dk, int dv, int chunk, int qkv_dtype,
                         bool g_scalar) {
    if (HK <= 0 || HV <= 0) return GDR_ERR_SHAPE;
    if (HV % HK != 0) return GDR_ERR_SHAPE;
    if (qkv_dtype != GDR_F32 && qkv_dtype != GDR_BF16) return GDR_ERR_UNSUPPORTED;
    if (!supported_dim(dk) || !supported_dim(dv) || !supported_chunk(chunk))
        return GDR_ERR_UNSUPPORTED;
    // every element count must fit comfortably in 63 bits, and grids in 31
    if (BT > (1LL << 40) || NS * HV > (1LL << 30)) return GDR_ERR_SHAPE;
    const bool work = BT > 0;
    if (work && (!q || !k || !v || !g || !beta || !out)) return GDR_ERR_NULL;
    // 16-byte alignment for everything read or written in vectors or bulk
    // copies; beta is only ever read one element at a time
    const void *ptrs[] = {q, k, v, g, h0, out, ht};
    for (const void *x : ptrs)
        if (x && !aligned16(x)) return GDR_ERR_ALIGN;
    if (beta && ((uintptr_t)beta & 3u) != 0) return GDR_ERR_ALIGN;

    const size_t es = qkv_dtype == GDR_BF16 ? 2 : 4;
    const Range rq = range_of(q, (size_t)BT * HK * dk * es);
    const Range rk = range_of(k, (size_t)BT * HK * dk * es);
    const Range rv = range_of(v, (size_t)BT * HV * dv * es);
    const Range rg = range_of(g, (size_t)BT * HV * (g_scalar ? 1 : dk) * 4);
    const Range rb = range_of(beta, (size_t)BT * HV * 4);
    const Range rs0 = h0 ? range_of(h0, (size_t)NS * HV * dk * dv * 4) : Range{0, 0};
    const Range ro = work ? range_of(out, (size_t)BT * HV * dv * es) : Range{0, 0};
    const Range rst = ht ? range_of(ht, (size_t)NS * HV * dk * dv * 4) : Range{0, 0};
    const Range ins[] = {rq, rk, rv, rg, rb};
    for (const Range &r : ins) {
        if (overlap(ro, r) || overlap(rst, r)) return GDR_ERR_ALIAS;
    }
    if (overlap(ro, rs0) || overlap(ro, rst)) return GDR_ERR_ALIAS;
    if (h0 && ht && h0 != ht && overlap(rs0, rst)) return GDR_ERR_ALIAS;
    return GDR_OK;
}

// Validates shapes and pointers of a dense [B, T] batch; fills `p`. Does not
// look at the workspace.
gdr_status validate(const void *q, const void *k, const void *v, const float *g,
                    const float *beta, const float *h0, void *out, float *ht, int B, int T,
                    int HK, int HV, int dk, int dv, int chunk, int qkv_dtype, gdr::Problem *p,
                    unsigned flags = 0) {
    if (B < 0 || T < 0) return GDR_ERR_SHAPE;
    const bool gs = (flags & GDR_FLAG_SCALAR_GATE) != 0;
    const gdr_status st = validate_rows(q, k, v, g, beta, h0, out, ht, (long long)B * T, B, HK,
                                        HV, dk, dv, chunk, qkv_dtype, gs);
    if (st != GDR_OK) return st;
    *p = gdr::Problem{q, k, v, g, beta, h0, out, ht, B, T, HK, HV, dk, dv, chunk,
                      qkv_dtype == GDR_BF16 ? 1 : 0, gs ? 1 : 0};
    return GDR_OK;
}

enum class Route {
    Nothing,
    EmptySequence,
    Decode,
    GenericPrefill,
    TensorCorePrefill,
    SegmentedPrefill
};

// `segments`: whether the tensor-core route may split the state scan into
// segments (dense batches only).
Route choose(const gdr::Problem &p, unsigned flags, bool segments = false) {
    if (p.B == 0) return Route::Nothing;
    if (p.T == 0) return Route::EmptySequence;
    if (p.T == 1 && !(flags & GDR_FLAG_FORCE_CHUNKED)) return Route::Decode;
    if (gdr::tc_prefill_supported(p) && !(flags & GDR_FLAG_FORCE_GENERIC)) {
        if (segments && (long long)p.B * p.T <= 0x7fffffffLL && gdr::segment_count(p, flags) >= 2)
            return Route::SegmentedPrefill;
        return Route::TensorCorePrefill;
    }
    return Route::GenericPrefill;
}

std::mutex g_err_mutex;
std::vector<int *> g_err_addr;

}  // namespace

namespace gdr {
// Device address of g_gdr_device_error on the current device (looked up once
// per device).
cudaError_t device_error_word(int **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_err_mutex);
    if ((int)g_err_addr.size() <= dev) g_err_addr.resize(dev + 1, nullptr);
    if (!g_err_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_gdr_device_error);
        if (e != cudaSuccess) return e;
        g_err_addr[dev] = static_cast<int *>(p);
    }
    *out = g_err_addr[dev];
    return cudaSuccess;
}
}  // namespace gdr

namespace {

size_t route_workspace(const gdr::Problem &p, Route r, unsigned flags) {
    if (r == Route::GenericPrefill)
        return gdr::generic_prefill_workspace_bytes(p, gdr::scan_segment_count(p, flags));
    if (r == Route::SegmentedPrefill)
        return gdr::segmented_workspace_bytes(p, gdr::segment_count(p, flags));
    return 0;
}

gdr_status run(const gdr::Problem &p, Route r, unsigned flags, void *ws, cudaStream_t stream) {
    cudaError_t e = cudaSuccess;
    switch (r) {
        case Route::Nothing:
            return GDR_OK;
        case Route::EmptySequence: {
            if (!p.ht) return GDR_OK;
            const size_t bytes = (size_t)p.B * p.HV * p.dk * p.dv * sizeof(float);
            if (p.h0 == p.ht) return GDR_OK;
            e = p.h0 ? cudaMemcpyAsync(p.ht, p.h0, bytes, cudaMemcpyDeviceToDevice, stream)
                     : cudaMemsetAsync(p.ht, 0, bytes, stream);
            break;
        }
        case Route::Decode:
            e = gdr::launch_decode(p, stream);
            break;
        case Route::GenericPrefill: {
            const bool tc = !(flags & GDR_FLAG_FORCE_GENERIC) && gdr::scan_tc_supported(p);
            e = gdr::launch_generic_prefill(p, ws, stream, tc,
                                            tc ? gdr::scan_segment_count(p, flags) : 0);
            break;
        }
        case Route::TensorCorePrefill: {
            int *err = nullptr;
            e = gdr::device_error_word(&err);
            if (e == cudaSuccess) e = gdr::launch_tc_prefill(p, err, stream);
            break;
        }
        case Route::SegmentedPrefill: {
            int *err = nullptr;
            e = gdr::device_error_word(&err);
            if (e == cudaSuccess)
                e = gdr::launch_segmented_prefill(p, gdr::segment_count(p, flags), ws, err, stream);
            break;
        }
    }
    return e == cudaSuccess ? GDR_OK : cuda_fail(e);
}

// ---- packed variable-length batches
//
// Workspace: the batch's tables (copied in from the host by one
// cudaMemcpyAsync), then the chunk records of the CUDA-core prefill.  Each
// part starts on a 256-byte boundary.
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct VarlenPlan {
    std::vector<int2> rows;      // single-token sequences: {token row, slot}
    std::vector<int4> tc_seqs;   // tensor-core prefill: {first row, length, slot, 0}
    std::vector<int4> gen_seqs;  // CUDA-core prefill: {first row, length, slot, first chunk}
    std::vector<int2> chunks;    // CUDA-core prefill: {first row, length} per chunk
    std::vector<int> empty;      // slots of zero-length sequences
    std::vector<gdr::SegSeq> seg_seqs;  // tensor-core prefill cut into seg_P segments
    int seg_P = 0;
    std::vector<gdr::ScanSeq> scan_seqs;  // chunk-record prefill cut into scan_P segments
    int scan_P = 0;
    size_t off_rows = 0, off_tc = 0, off_maps = 0, off_gen = 0, off_chunks = 0;
    size_t table_bytes = 0, record_off = 0, off_seg = 0, off_scan = 0, total_bytes = 0;
};

// Checks cu_seqlens (cu[0] = 0, non-decreasing, cu[N] < 2^31) and assigns
// every sequence its route.  `p` carries the shapes; its pointers may be null.
gdr_status check_cu_seqlens(const int *cu, int N) {
    if (N < 0) return GDR_ERR_SHAPE;
    if (N > 0 && !cu) return GDR_ERR_NULL;
    if (N > 0 && cu[0] != 0) return GDR_ERR_SHAPE;
    for (int n = 0; n < N; ++n)
        if (cu[n + 1] < cu[n]) return GDR_ERR_SHAPE;
    return GDR_OK;
}

gdr_status plan_varlen(const int *cu, int N, const gdr::Problem &p, unsigned flags,
                       VarlenPlan *plan) {
    const gdr_status st = check_cu_seqlens(cu, N);
    if (st != GDR_OK) return st;
    gdr::Problem one = p;  // a sequence of length L, for routing
    one.B = 1;
    long long nch = 0;
    for (int n = 0; n < N; ++n) {
        const int L = cu[n + 1] - cu[n];
        one.T = L;
        switch (choose(one, flags)) {
            case Route::Nothing:
                break;
            case Route::EmptySequence:
                plan->empty.push_back(n);
                break;
            case Route::Decode:
                plan->rows.push_back(make_int2(cu[n], n));
                break;
            case Route::TensorCorePrefill:
            case Route::SegmentedPrefill:  // not chosen here
                plan->tc_seqs.push_back(make_int4(cu[n], L, n, 0));
                break;
            case Route::GenericPrefill:
                plan->gen_seqs.push_back(make_int4(cu[n], L, n, 0));
                nch += (L + p.chunk - 1) / p.chunk;
                break;
        }
    }
    if (nch * p.HV > 0x7fffffffLL) return GDR_ERR_SHAPE;
    // longest first: a sequence's CTAs run its chunks in order, so the long
    // ones start at once and the short ones fill in behind them
    auto longer = [](const int4 &a, const int4 &b) { return a.y > b.y; };
    std::stable_sort(plan->tc_seqs.begin(), plan->tc_seqs.end(), longer);
    std::stable_sort(plan->gen_seqs.begin(), plan->gen_seqs.end(), longer);
    // long tensor-core sequences on an otherwise idle device: cut into
    // segments (the chunk-parallel state scan); the others walk whole
    if (!plan->tc_seqs.empty()) {
        std::vector<int> lengths;
        for (const int4 &sd : plan->tc_seqs) lengths.push_back(sd.y);
        std::vector<char> cut;
        const int P = gdr::varlen_segment_count(p, lengths.data(), (int)lengths.size(), flags, &cut);
        if (P >= 2) {
            std::vector<int4> walk;
            for (size_t i = 0; i < plan->tc_seqs.size(); ++i) {
                const int4 sd = plan->tc_seqs[i];
                if (cut[i])
                    plan->seg_seqs.push_back(gdr::SegSeq{(size_t)sd.x, sd.y, sd.z});
                else
                    walk.push_back(sd);
            }
            plan->tc_seqs.swap(walk);
            plan->seg_P = P;
        }
    }
    for (int4 &sd : plan->gen_seqs) {
        sd.w = (int)plan->chunks.size();
        for (int t = 0; t < sd.y; t += p.chunk)
            plan->chunks.push_back(make_int2(sd.x + t, std::min(p.chunk, sd.y - t)));
    }
    // the same for long sequences on the chunk-record route: every chunk's
    // record is written at once, the cut ones' state scans run in segments
    if (!plan->gen_seqs.empty()) {
        std::vector<int> lengths;
        for (const int4 &sd : plan->gen_seqs) lengths.push_back(sd.y);
        std::vector<char> cut;
        const int P =
            gdr::scan_varlen_segment_count(p, lengths.data(), (int)lengths.size(), flags, &cut);
        if (P >= 2) {
            std::vector<int4> walk;
            for (size_t i = 0; i < plan->gen_seqs.size(); ++i) {
                const int4 sd = plan->gen_seqs[i];
                if (cut[i])
                    plan->scan_seqs.push_back(
                        gdr::ScanSeq{sd.x, (long long)sd.w * p.HV, sd.y, sd.z, 1, p.HV});
                else
                    walk.push_back(sd);
            }
            plan->gen_seqs.swap(walk);
            plan->scan_P = P;
        }
    }
    size_t off = 0;
    plan->off_rows = off;
    off = align256(off + plan->rows.size() * sizeof(int2));
    plan->off_tc = off;
    off = align256(off + plan->tc_seqs.size() * sizeof(int4));
    plan->off_maps = off;
    off = align256(off + plan->tc_seqs.size() * gdr::tc_seq_maps_bytes());
    plan->off_gen = off;
    off = align256(off + plan->gen_seqs.size() * sizeof(int4));
    plan->off_chunks = off;
    off = align256(off + plan->chunks.size() * sizeof(int2));
    plan->table_bytes = off;
    plan->record_off = off;
    const bool any = !plan->rows.empty() || !plan->tc_seqs.empty() || !plan->gen_seqs.empty() ||
                     !plan->seg_seqs.empty() || !plan->scan_seqs.empty();
    plan->total_bytes =
        any ? off + gdr::generic_varlen_record_bytes(p, (long long)plan->chunks.size()) : 0;
    if (!plan->seg_seqs.empty()) {
        plan->off_seg = align256(plan->total_bytes);
        plan->total_bytes = plan->off_seg + gdr::segmented_list_workspace_bytes(
                                                p, (int)plan->seg_seqs.size(), plan->seg_P);
    }
    if (!plan->scan_seqs.empty()) {
        plan->off_scan = align256(plan->total_bytes);
        plan->total_bytes = plan->off_scan + gdr::scan_segmented_bytes(
                                                 p, (int)plan->scan_seqs.size(), plan->scan_P);
    }
    return GDR_OK;
}

// gdr_forward's workspace, one per device: the caller's (gdr_set_workspace)
// when registered, else the library's own, grown on demand.
struct OwnedWorkspace {
    void *ptr = nullptr;   // library-owned
    size_t bytes = 0;
    void *user = nullptr;  // caller-owned, registered
    size_t user_bytes = 0;
};
std::mutex g_ws_mutex;
std::vector<OwnedWorkspace> g_ws;

// ---- launch tracing: a pair of CUDA events on the launching stream around
// every kernel launch of this library, while enabled.
struct TraceRec {
    int kernel;
    cudaEvent_t a, b;
};
std::mutex g_trace_mutex;
bool g_trace_on = false;
std::vector<TraceRec> g_trace;
std::vector<cudaEvent_t> g_event_pool;
thread_local cudaEvent_t t_pending_begin = nullptr;

cudaEvent_t take_event() {
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

const char *kKernelNames[gdr::kNumKernels] = {"gdr_decode_kernel", "gdr_chunk_prep",
                                              "gdr_chunk_scan",    "gdr_prefill_fused",
                                              "gdr_segment_init",  "gdr_segment_combine",
                                              "gdr_tree_tc",       "gdr_tree_path_kernel",
                                              "gdr_tree_gram_kernel", "gdr_tree_solve_kernel",
                                              "gdr_chunk_scan_tc", "gdr_chunk_prep_tc"};

}  // namespace

namespace gdr {
// Lets other translation units of the library report a CUDA failure through
// gdr_last_cuda_error().
int record_cuda_error(cudaError_t e) {
    t_last_cuda_error = (int)e;
    return (int)e;
}

void trace_begin(int kernel, cudaStream_t stream) {
    (void)kernel;
    std::lock_guard<std::mutex> lock(g_trace_mutex);
    if (!g_trace_on) return;
    cudaEvent_t e = take_event();
    if (e && cudaEventRecord(e, stream) == cudaSuccess) t_pending_begin = e;
}
void trace_end(int kernel, cudaStream_t stream) {
    std::lock_guard<std::mutex> lock(g_trace_mutex);
    if (!g_trace_on || !t_pending_begin) return;
    cudaEvent_t e = take_event();
    if (e && cudaEventRecord(e, stream) == cudaSuccess) {
        g_trace.push_back(TraceRec{kernel, t_pending_begin, e});
    }
    t_pending_begin = nullptr;
}
}  // namespace gdr

namespace {
// Trees run as one chunk of the CUDA-core kernels: the smallest supported
// chunk that holds T tokens (0 when T is too large).
int tree_chunk(int T) { return T <= 16 ? 16 : T <= 32 ? 32 : T <= 64 ? 64 : 0; }
constexpr int kTreeMaxTokens = 512;

bool tree_on_tensor_cores(const gdr::Problem &p, unsigned flags) {
    gdr::Problem c = p;
    c.chunk = 64;
    return gdr::tc_prefill_supported(c) && !(flags & GDR_FLAG_FORCE_GENERIC) &&
           !(flags & GDR_FLAG_SCALAR_GATE);
}

// Trees past one chunk, or any with GDR_FLAG_TREE_BLOCKED, take the blocked
// solve.
bool tree_blocked(const gdr::Problem &p, unsigned flags) {
    return p.T > 64 || (flags & GDR_FLAG_TREE_BLOCKED);
}
// The Problem of a tree call: the chunk of the one-chunk routes (64 on the
// blocked route, where it plays no part).
int tree_problem_chunk(int T, unsigned flags) {
    return (T > 64 || (flags & GDR_FLAG_TREE_BLOCKED)) ? 64 : tree_chunk(T > 0 ? T : 1);
}

// Workspace: the parents, then the route's own: the per-tree records (CUDA-core
// route) or the ancestor masks and path sums (blocked route).
size_t tree_layout(const gdr::Problem &p, unsigned flags, size_t *record_off) {
    const size_t table = align256((size_t)p.B * p.T * sizeof(int));
    *record_off = table;
    if (tree_blocked(p, flags)) return table + gdr::tree_blocked_workspace_bytes(p);
    return table + (tree_on_tensor_cores(p, flags) ? 0 : gdr::generic_tree_record_bytes(p));
}
}  // namespace

extern "C" {

GDR_API gdr_status gdr_trace_enable(int on) {
    std::lock_guard<std::mutex> lock(g_trace_mutex);
    g_trace_on = on != 0;
    return GDR_OK;
}

GDR_API int gdr_trace_read(int max_kernels, const char **names, int *launches, double *total_ms) {
    std::vector<TraceRec> recs;
    {
        std::lock_guard<std::mutex> lock(g_trace_mutex);
        recs.swap(g_trace);
    }
    const int n = max_kernels < gdr::kNumKernels ? max_kernels : gdr::kNumKernels;
    for (int i = 0; i < n; ++i) {
        if (names) names[i] = kKernelNames[i];
        if (launches) launches[i] = 0;
        if (total_ms) total_ms[i] = 0.0;
    }
    int status = 0;
    for (const TraceRec &r : recs) {
        float ms = 0.f;
        if (cudaEventSynchronize(r.b) != cudaSuccess ||
            cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess)
            status = -1;
        if (r.kernel < n) {
            if (launches) launches[r.kernel] += 1;
            if (total_ms) total_ms[r.kernel] += ms;
        }
    }
    std::lock_guard<std::mutex> lock(g_trace_mutex);
    for (const TraceRec &r : recs) {
        g_event_pool.push_back(r.a);
        g_event_pool.push_back(r.b);
    }
    return status < 0 ? status : n;
}

GDR_API size_t gdr_workspace_bytes(int B, int T, int HK, int HV, int dk, int dv, int chunk,
                                   int qkv_dtype, unsigned flags) {
    // shape-only validation: use a fake aligned, non-overlapping pointer set
    gdr::Problem p;
    if (B < 0 || T < 0 || HK <= 0 || HV <= 0 || HV % HK != 0) return 0;
    if (qkv_dtype != GDR_F32 && qkv_dtype != GDR_BF16) return 0;
    if (!supported_dim(dk) || !supported_dim(dv) || !supported_chunk(chunk)) return 0;
    p = gdr::Problem{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                     B, T, HK, HV, dk, dv, chunk, qkv_dtype == GDR_BF16 ? 1 : 0,
                     (flags & GDR_FLAG_SCALAR_GATE) ? 1 : 0};
    return route_workspace(p, choose(p, flags, true), flags);
}

GDR_API gdr_status gdr_forward_ex(const void *q, const void *k, const void *v, const float *g,
                                  const float *beta, const float *h0, void *out, float *ht,
                                  int B, int T, int HK, int HV, int dk, int dv, int chunk,
                                  void *stream, int qkv_dtype, void *workspace,
                                  size_t workspace_bytes, unsigned flags) {
    gdr::Problem p;
    gdr_status st = validate(q, k, v, g, beta, h0, out, ht, B, T, HK, HV, dk, dv, chunk,
                             qkv_dtype, &p, flags);
    if (st != GDR_OK) return st;
    const Route r = choose(p, flags, true);
    const size_t need = route_workspace(p, r, flags);
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return GDR_ERR_WORKSPACE;
        if (((uintptr_t)workspace & 255u) != 0) return GDR_ERR_ALIGN;
    }
    return run(p, r, flags, workspace, static_cast<cudaStream_t>(stream));
}

GDR_API gdr_status gdr_forward(const void *q, const void *k, const void *v, const float *g,
                               const float *beta, const float *h0, void *out, float *ht, int B,
                               int T, int HK, int HV, int dk, int dv, int chunk, void *stream,
                               int qkv_dtype) {
    gdr::Problem p;
    gdr_status st = validate(q, k, v, g, beta, h0, out, ht, B, T, HK, HV, dk, dv, chunk,
                             qkv_dtype, &p);
    if (st != GDR_OK) return st;
    const Route r = choose(p, 0u, true);
    const size_t need = route_workspace(p, r, 0u);
    void *ws = nullptr;
    if (need > 0) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return cuda_fail(e);
        std::lock_guard<std::mutex> lock(g_ws_mutex);
        if ((int)g_ws.size() <= dev) g_ws.resize(dev + 1);
        OwnedWorkspace &w = g_ws[dev];
        if (w.user) {
            if (w.user_bytes < need) return GDR_ERR_WORKSPACE;
            ws = w.user;
        } else if (w.bytes < need) {
            if (w.ptr) {
                // the old buffer may still be in use by earlier launches
                e = cudaDeviceSynchronize();
                if (e != cudaSuccess) return cuda_fail(e);
                cudaFree(w.ptr);
                w.ptr = nullptr;
                w.bytes = 0;
            }
            e = cudaMalloc(&w.ptr, need);
            if (e != cudaSuccess) return cuda_fail(e);
            w.bytes = need;
        }
        if (!ws) ws = w.ptr;
    }
    return run(p, r, 0u, ws, static_cast<cudaStream_t>(stream));
}

GDR_API gdr_status gdr_set_workspace(void *dev_ptr, size_t bytes) {
    if (bytes > 0 && !dev_ptr) return GDR_ERR_NULL;
    if (dev_ptr && ((uintptr_t)dev_ptr & 255u) != 0) return GDR_ERR_ALIGN;
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    if ((int)g_ws.size() <= dev) g_ws.resize(dev + 1);
    g_ws[dev].user = (dev_ptr && bytes > 0) ? dev_ptr : nullptr;
    g_ws[dev].user_bytes = g_ws[dev].user ? bytes : 0;
    return GDR_OK;
}

GDR_API size_t gdr_varlen_workspace_bytes(const int *cu_seqlens, int N, int HK, int HV, int dk,
                                          int dv, int chunk, int qkv_dtype, unsigned flags) {
    if (HK <= 0 || HV <= 0 || HV % HK != 0) return 0;
    if (qkv_dtype != GDR_F32 && qkv_dtype != GDR_BF16) return 0;
    if (!supported_dim(dk) || !supported_dim(dv) || !supported_chunk(chunk)) return 0;
    const gdr::Problem p{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                         N, 0, HK, HV, dk, dv, chunk, qkv_dtype == GDR_BF16 ? 1 : 0};
    VarlenPlan plan;
    if (plan_varlen(cu_seqlens, N, p, flags, &plan) != GDR_OK) return 0;
    return plan.total_bytes;
}

GDR_API gdr_status gdr_forward_varlen(const void *q, const void *k, const void *v, const float *g,
                                      const float *beta, const float *h0, void *out, float *ht,
                                      const int *cu_seqlens, int N, int HK, int HV, int dk, int dv,
                                      int chunk, void *stream, int qkv_dtype, void *workspace,
                                      size_t workspace_bytes, unsigned flags) {
    gdr_status st = check_cu_seqlens(cu_seqlens, N);
    if (st != GDR_OK) return st;
    const long long total = N > 0 ? cu_seqlens[N] : 0;
    const bool gs = (flags & GDR_FLAG_SCALAR_GATE) != 0;
    st = validate_rows(q, k, v, g, beta, h0, out, ht, total, N, HK, HV, dk, dv, chunk,
                                  qkv_dtype, gs);
    if (st != GDR_OK) return st;
    const gdr::Problem base{q, k, v, g, beta, h0, out, ht, N, 0, HK, HV, dk, dv, chunk,
                            qkv_dtype == GDR_BF16 ? 1 : 0, gs ? 1 : 0};
    VarlenPlan plan;
    st = plan_varlen(cu_seqlens, N, base, flags, &plan);
    if (st != GDR_OK) return st;
    if (plan.total_bytes > 0) {
        if (!workspace || workspace_bytes < plan.total_bytes) return GDR_ERR_WORKSPACE;
        if (((uintptr_t)workspace & 255u) != 0) return GDR_ERR_ALIGN;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    cudaError_t e = cudaSuccess;

    // tables, staged on the host and copied in one piece
    if (plan.table_bytes > 0) {
        std::vector<unsigned char> host(plan.table_bytes, 0);
        if (!plan.rows.empty())
            memcpy(host.data() + plan.off_rows, plan.rows.data(), plan.rows.size() * sizeof(int2));
        if (!plan.tc_seqs.empty())
            memcpy(host.data() + plan.off_tc, plan.tc_seqs.data(), plan.tc_seqs.size() * sizeof(int4));
        for (size_t i = 0; i < plan.tc_seqs.size(); ++i) {
            e = gdr::tc_encode_seq_maps(base, (size_t)plan.tc_seqs[i].x, plan.tc_seqs[i].y,
                                        host.data() + plan.off_maps + i * gdr::tc_seq_maps_bytes());
            if (e != cudaSuccess) return cuda_fail(e);
        }
        if (!plan.gen_seqs.empty())
            memcpy(host.data() + plan.off_gen, plan.gen_seqs.data(), plan.gen_seqs.size() * sizeof(int4));
        if (!plan.chunks.empty())
            memcpy(host.data() + plan.off_chunks, plan.chunks.data(), plan.chunks.size() * sizeof(int2));
        // pageable source: the call returns once the bytes have been taken
        e = cudaMemcpyAsync(ws, host.data(), plan.table_bytes, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    // zero-length sequences: the final state is the initial one
    if (ht && h0 != ht) {
        const size_t bytes = (size_t)HV * dk * dv * sizeof(float);
        for (int n : plan.empty) {
            float *dst = ht + (size_t)n * HV * dk * dv;
            e = h0 ? cudaMemcpyAsync(dst, h0 + (size_t)n * HV * dk * dv, bytes,
                                     cudaMemcpyDeviceToDevice, s)
                   : cudaMemsetAsync(dst, 0, bytes, s);
            if (e != cudaSuccess) return cuda_fail(e);
        }
    }
    if (!plan.rows.empty()) {
        gdr::Problem p = base;
        p.B = (int)plan.rows.size();
        p.T = 1;
        e = gdr::launch_decode_rows(p, reinterpret_cast<const int2 *>(ws + plan.off_rows), s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (!plan.tc_seqs.empty()) {
        int *err = nullptr;
        e = gdr::device_error_word(&err);
        if (e != cudaSuccess) return cuda_fail(e);
        gdr::Problem p = base;
        p.B = (int)plan.tc_seqs.size();
        e = gdr::launch_tc_prefill_varlen(p, ws + plan.off_maps,
                                          reinterpret_cast<const int4 *>(ws + plan.off_tc), p.B,
                                          err, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (!plan.seg_seqs.empty()) {
        int *err = nullptr;
        e = gdr::device_error_word(&err);
        if (e != cudaSuccess) return cuda_fail(e);
        e = gdr::launch_segmented_list(base, plan.seg_seqs.data(), (int)plan.seg_seqs.size(),
                                       plan.seg_P, ws + plan.off_seg, err, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (!plan.gen_seqs.empty() || !plan.scan_seqs.empty()) {
        gdr::Problem p = base;
        p.B = (int)plan.gen_seqs.size();
        e = gdr::launch_generic_prefill_varlen(
            p, ws + plan.record_off, reinterpret_cast<const int2 *>(ws + plan.off_chunks),
            (int)plan.chunks.size(), reinterpret_cast<const int4 *>(ws + plan.off_gen), s,
            !(flags & GDR_FLAG_FORCE_GENERIC) && gdr::scan_tc_supported(p),
            plan.scan_seqs.data(), (int)plan.scan_seqs.size(), plan.scan_P, ws + plan.off_scan);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return GDR_OK;
}

GDR_API size_t gdr_tree_workspace_bytes(int B, int T, int HK, int HV, int dk, int dv,
                                        int qkv_dtype, unsigned flags) {
    if (B < 0 || T < 0 || HK <= 0 || HV <= 0 || HV % HK != 0) return 0;
    if (qkv_dtype != GDR_F32 && qkv_dtype != GDR_BF16) return 0;
    if (!supported_dim(dk) || !supported_dim(dv) || T > kTreeMaxTokens) return 0;
    if ((long long)B * T == 0) return 0;
    const gdr::Problem p{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                         B, T, HK, HV, dk, dv, tree_problem_chunk(T, flags),
                         qkv_dtype == GDR_BF16 ? 1 : 0, (flags & GDR_FLAG_SCALAR_GATE) ? 1 : 0};
    size_t off = 0;
    return tree_layout(p, flags, &off);
}

GDR_API gdr_status gdr_forward_tree(const void *q, const void *k, const void *v, const float *g,
                                    const float *beta, const float *h0, void *out,
                                    const int *parent, int B, int T, int HK, int HV, int dk,
                                    int dv, void *stream, int qkv_dtype, void *workspace,
                                    size_t workspace_bytes, unsigned flags) {
    if (B < 0 || T < 0) return GDR_ERR_SHAPE;
    if (T > kTreeMaxTokens) return GDR_ERR_UNSUPPORTED;
    const int chunk = tree_problem_chunk(T, flags);
    gdr::Problem p;
    gdr_status st = validate(q, k, v, g, beta, h0, out, nullptr, B, T, HK, HV, dk, dv, chunk,
                             qkv_dtype, &p, flags);
    if (st != GDR_OK) return st;
    if ((long long)B * T == 0) return GDR_OK;
    if (!parent) return GDR_ERR_NULL;
    for (long long bt = 0; bt < (long long)B * T; ++bt) {
        const int t = (int)(bt % T);
        if (parent[bt] < -1 || parent[bt] >= t) return GDR_ERR_SHAPE;
    }
    size_t record_off = 0;
    const size_t need = tree_layout(p, flags, &record_off);
    if (!workspace || workspace_bytes < need) return GDR_ERR_WORKSPACE;
    if (((uintptr_t)workspace & 255u) != 0) return GDR_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    // the parents, from pageable host memory: taken before the call returns
    cudaError_t e = cudaMemcpyAsync(ws, parent, (size_t)B * T * sizeof(int),
                                    cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e);
    const int *par_dev = reinterpret_cast<const int *>(ws);
    if (tree_blocked(p, flags)) {
        if (!gdr::tree_blocked_supported(p)) return GDR_ERR_UNSUPPORTED;
        e = gdr::launch_tree_blocked(
            p, ws + record_off, par_dev,
            (flags & GDR_FLAG_TREE_GRAM_PER_VALUE_HEAD) ? gdr::kTreeGramPerValueHead : 0u, s);
    } else if (tree_on_tensor_cores(p, flags)) {
        int *err = nullptr;
        e = gdr::device_error_word(&err);
        if (e == cudaSuccess) {
            gdr::Problem tc = p;
            tc.chunk = 64;
            e = gdr::launch_tc_tree(tc, par_dev, err, s);
        }
    } else {
        e = gdr::launch_generic_tree(p, ws + record_off, par_dev, s);
    }
    return e == cudaSuccess ? GDR_OK : cuda_fail(e);
}

GDR_API gdr_status gdr_device_check(void *stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    int word = 0;
    e = cudaMemcpyFromSymbol(&word, g_gdr_device_error, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e);
    if (word != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_gdr_device_error, &zero, sizeof(int));
        if (e != cudaSuccess) return cuda_fail(e);
        return GDR_ERR_TIMEOUT;
    }
    return GDR_OK;
}

GDR_API const char *gdr_status_string(int status) {
    switch (status) {
        case GDR_OK: return "GDR_OK";
        case GDR_ERR_NULL: return "GDR_ERR_NULL: a required pointer is NULL";
        case GDR_ERR_SHAPE: return "GDR_ERR_SHAPE: invalid or overflowing shape (or HV % HK != 0)";
        case GDR_ERR_UNSUPPORTED: return "GDR_ERR_UNSUPPORTED: dk, dv, chunk or dtype not supported";
        case GDR_ERR_ALIGN: return "GDR_ERR_ALIGN: pointer not 16-byte aligned (workspace: 256)";
        case GDR_ERR_WORKSPACE: return "GDR_ERR_WORKSPACE: workspace missing or too small";
        case GDR_ERR_CUDA: return "GDR_ERR_CUDA: a CUDA call or launch failed";
        case GDR_ERR_TIMEOUT: return "GDR_ERR_TIMEOUT: a kernel gave up on a bounded wait";
        case GDR_ERR_ALIAS: return "GDR_ERR_ALIAS: an output overlaps another argument";
        default: return "unknown gdr_status";
    }
}

GDR_API int gdr_last_cuda_error(void) { return t_last_cuda_error; }

GDR_API const char *gdr_version(void) { return "0.1.0"; }

}  // extern "C"
