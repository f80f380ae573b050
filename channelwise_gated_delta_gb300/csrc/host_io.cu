// host_io.cu -- gdr_forward_host: the forward pass on HOST buffers, with the
// host-to-device copies, the compute and the device-to-host copies overlapped.
//
// The link between host and device memory is the bound, so the aim is to
// keep the copy-in stream busy from the first byte to the last and to start
// computing as soon as possible.  The recurrence over a sequence can stop
// after any token and resume from the state it reached, so every batch
// element is streamed in segments of whole chunks: segment s of element b
// runs as a B = 1 call that starts from the state segment s - 1 left in a
// device state buffer (h0[b] copied in for s = 0) and leaves its own there.
// Two device slots hold the inputs and outputs of two segments: while one
// segment computes on the caller's stream, the next is copied in on a
// copy-in stream and the previous one's output copied out on a copy-out
// stream.  Two state buffers let the first segment of the next element copy
// its h0 in while the current element still runs.
#include <mutex>
#include <stdint.h>
#include <vector>

#include "common.cuh"
#include "gdr.h"

namespace {

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Tokens per segment: a multiple of the chunk length, so that segmenting
// keeps every chunk of the unsegmented call; whole sequences up to twice it.
constexpr int kSegmentTokens = 2048;

int segment_tokens(int T, int chunk) {
    if (T <= 2 * kSegmentTokens) return T;
    return (kSegmentTokens / chunk) * chunk;
}

// The segmented state scan copies its tables from pageable host memory, which
// may wait for the compute stream and so stall the copy pipeline; the host
// entry is bound by its copies anyway.
constexpr unsigned kSegFlags = GDR_FLAG_NO_SEGMENTS;

// Per-slot layout: one segment's inputs, output and route workspace.
struct SlotLayout {
    size_t q, k, v, g, beta, out, ws, bytes;  // offsets and slot size
    size_t tq, tv, tg, tb;                     // bytes per token
    size_t ws_b;                               // route workspace bytes
};

SlotLayout slot_layout(int Ts, int HK, int HV, int dk, int dv, int chunk, int qkv_dtype) {
    SlotLayout L{};
    const size_t es = qkv_dtype == GDR_BF16 ? 2 : 4;
    L.tq = (size_t)HK * dk * es;
    L.tv = (size_t)HV * dv * es;
    L.tg = (size_t)HV * dk * 4;
    L.tb = (size_t)HV * 4;
    L.ws_b = gdr_workspace_bytes(1, Ts, HK, HV, dk, dv, chunk, qkv_dtype, kSegFlags);
    size_t off = 0;
    auto put = [&](size_t n) {
        const size_t at = off;
        off = align256(off + n);
        return at;
    };
    L.q = put(Ts * L.tq);
    L.k = put(Ts * L.tq);
    L.v = put(Ts * L.tv);
    L.g = put(Ts * L.tg);
    L.beta = put(Ts * L.tb);
    L.out = put(Ts * L.tv);
    L.ws = put(L.ws_b);
    L.bytes = off;
    return L;
}

constexpr int kSlots = 2;

// Library-owned copy streams and events, one set per device.
struct DeviceIo {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr;
    cudaEvent_t join_in = nullptr, join_out = nullptr;  // error paths: side streams -> caller
    cudaEvent_t in_ready[kSlots] = {}, computed[kSlots] = {}, out_done[kSlots] = {};
    cudaEvent_t state_done[kSlots] = {};
};
std::mutex g_io_mutex;
std::vector<DeviceIo> g_io;

cudaError_t device_io(DeviceIo **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((int)g_io.size() <= dev) g_io.resize(dev + 1);
    DeviceIo &io = g_io[dev];
    if (!io.ready) {
        const unsigned ef = cudaEventDisableTiming;
        e = cudaStreamCreateWithFlags(&io.in, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&io.out, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&io.start, ef);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&io.join_in, ef);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&io.join_out, ef);
        for (int s = 0; s < kSlots && e == cudaSuccess; ++s) {
            e = cudaEventCreateWithFlags(&io.in_ready[s], ef);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&io.computed[s], ef);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&io.out_done[s], ef);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&io.state_done[s], ef);
        }
        if (e != cudaSuccess) return e;
        io.ready = true;
    }
    *out = &io;
    return cudaSuccess;
}

bool valid_shape(int B, int T, int HK, int HV, int dk, int dv, int chunk, int qkv_dtype) {
    auto dim_ok = [](int d) { return d == 32 || d == 64 || d == 128; };
    return B >= 0 && T >= 0 && HK > 0 && HV > 0 && HV % HK == 0 && dim_ok(dk) && dim_ok(dv) &&
           (chunk == 16 || chunk == 32 || chunk == 64) &&
           (qkv_dtype == GDR_F32 || qkv_dtype == GDR_BF16) &&
           (long long)B * T <= (1LL << 40);
}

size_t state_bytes(int HV, int dk, int dv) { return (size_t)HV * dk * dv * 4; }

int segments_per_element(int T, int Ts) { return T == 0 ? 1 : (T + Ts - 1) / Ts; }

// Staging: the slots (two, or one per segment if fewer), then the state
// buffers (two, or one per batch element if fewer).
struct Staging {
    int slots, states;
    size_t bytes;
};
Staging staging_plan(int B, int T, int HK, int HV, int dk, int dv, int chunk, int qkv_dtype) {
    const int Ts = segment_tokens(T, chunk);
    const SlotLayout L = slot_layout(Ts, HK, HV, dk, dv, chunk, qkv_dtype);
    const long long segs_total = (long long)B * segments_per_element(T, Ts);
    Staging p;
    p.slots = segs_total < kSlots ? (int)segs_total : kSlots;
    p.states = B < kSlots ? B : kSlots;
    p.bytes = (size_t)p.slots * L.bytes + (size_t)p.states * align256(state_bytes(HV, dk, dv));
    return p;
}

}  // namespace

extern "C" {

GDR_API size_t gdr_host_staging_bytes(int B, int T, int HK, int HV, int dk, int dv, int chunk,
                                      int qkv_dtype) {
    if (!valid_shape(B, T, HK, HV, dk, dv, chunk, qkv_dtype) || B == 0) return 0;
    return staging_plan(B, T, HK, HV, dk, dv, chunk, qkv_dtype).bytes;
}

GDR_API gdr_status gdr_forward_host(const void *q, const void *k, const void *v, const float *g,
                                    const float *beta, const float *h0, void *out, float *ht,
                                    int B, int T, int HK, int HV, int dk, int dv, int chunk,
                                    void *stream, int qkv_dtype, void *staging,
                                    size_t staging_bytes_given) {
    if (!valid_shape(B, T, HK, HV, dk, dv, chunk, qkv_dtype)) {
        if (B < 0 || T < 0 || HK <= 0 || HV <= 0 || HV % HK != 0) return GDR_ERR_SHAPE;
        return GDR_ERR_UNSUPPORTED;
    }
    if (B == 0) return GDR_OK;
    if ((long long)T > 0 && (!q || !k || !v || !g || !beta || !out)) return GDR_ERR_NULL;
    const int Ts = segment_tokens(T, chunk);
    const SlotLayout L = slot_layout(Ts, HK, HV, dk, dv, chunk, qkv_dtype);
    const Staging plan = staging_plan(B, T, HK, HV, dk, dv, chunk, qkv_dtype);
    if (!staging || staging_bytes_given < plan.bytes) return GDR_ERR_WORKSPACE;
    if (((uintptr_t)staging & 255u) != 0) return GDR_ERR_ALIGN;
    const size_t sb = state_bytes(HV, dk, dv);
    char *state_base = static_cast<char *>(staging) + (size_t)plan.slots * L.bytes;

    std::lock_guard<std::mutex> lock(g_io_mutex);
    DeviceIo *io = nullptr;
    cudaError_t e = device_io(&io);
    if (e != cudaSuccess) {
        gdr::record_cuda_error(e);
        return GDR_ERR_CUDA;
    }
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // Once copies have been queued on the library's side streams, an error
    // return must not leave them running behind the caller's back: they read
    // and write the caller's host buffers and this call's staging.  The
    // caller's stream is made to wait for both side streams (or, if that
    // cannot be queued, the side streams are drained on the host) before the
    // error is reported, so the caller may free or reuse its buffers once its
    // own stream has completed.
    bool queued = false;
    auto join = [&]() {
        if (!queued) return;
        const bool ok = cudaEventRecord(io->join_in, io->in) == cudaSuccess &&
                        cudaEventRecord(io->join_out, io->out) == cudaSuccess &&
                        cudaStreamWaitEvent(cs, io->join_in, 0) == cudaSuccess &&
                        cudaStreamWaitEvent(cs, io->join_out, 0) == cudaSuccess;
        if (!ok) {
            cudaStreamSynchronize(io->in);
            cudaStreamSynchronize(io->out);
        }
    };
    auto fail = [&](cudaError_t err) {
        gdr::record_cuda_error(err);
        join();
        return GDR_ERR_CUDA;
    };
    // everything earlier on the caller's stream comes first
    if ((e = cudaEventRecord(io->start, cs)) != cudaSuccess) return fail(e);
    queued = true;
    if ((e = cudaStreamWaitEvent(io->in, io->start, 0)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamWaitEvent(io->out, io->start, 0)) != cudaSuccess) return fail(e);

    const char *hq = static_cast<const char *>(q), *hk = static_cast<const char *>(k);
    const char *hv = static_cast<const char *>(v);
    const char *hg = reinterpret_cast<const char *>(g), *hb = reinterpret_cast<const char *>(beta);
    const char *hs = reinterpret_cast<const char *>(h0);
    char *ho = static_cast<char *>(out), *hh = reinterpret_cast<char *>(ht);
    const int nseg = segments_per_element(T, Ts);
    int n = 0;  // segments issued so far
    for (int b = 0; b < B; ++b) {
        const int st = b % kSlots;
        float *state = reinterpret_cast<float *>(state_base + (size_t)st * align256(sb));
        for (int s = 0; s < nseg; ++s, ++n) {
            const int slot = n % kSlots;
            const size_t t0 = (size_t)s * Ts;
            const int len = T == 0 ? 0 : (int)((size_t)T - t0 < (size_t)Ts ? T - t0 : Ts);
            const size_t row0 = (size_t)b * T + t0;  // first token row in the host tensors
            char *sl = static_cast<char *>(staging) + (size_t)slot * L.bytes;
            // the slot is free once the copies out of its previous segment are done
            if (n >= kSlots && (e = cudaStreamWaitEvent(io->in, io->out_done[slot], 0)) != cudaSuccess)
                return fail(e);
            struct Copy {
                char *dst;
                const char *src;
                size_t n;
            } ins[] = {{sl + L.q, hq + row0 * L.tq, len * L.tq},
                       {sl + L.k, hk + row0 * L.tq, len * L.tq},
                       {sl + L.v, hv + row0 * L.tv, len * L.tv},
                       {sl + L.g, hg + row0 * L.tg, len * L.tg},
                       {sl + L.beta, hb + row0 * L.tb, len * L.tb}};
            if (s == 0 && hs) {
                // the state buffer is free once the element two back left it
                if (b >= kSlots &&
                    (e = cudaStreamWaitEvent(io->in, io->state_done[st], 0)) != cudaSuccess)
                    return fail(e);
                e = cudaMemcpyAsync(state, hs + (size_t)b * sb, sb, cudaMemcpyHostToDevice, io->in);
                if (e != cudaSuccess) return fail(e);
            }
            for (const Copy &c : ins) {
                if (c.n == 0) continue;
                e = cudaMemcpyAsync(c.dst, c.src, c.n, cudaMemcpyHostToDevice, io->in);
                if (e != cudaSuccess) return fail(e);
            }
            if ((e = cudaEventRecord(io->in_ready[slot], io->in)) != cudaSuccess) return fail(e);
            if ((e = cudaStreamWaitEvent(cs, io->in_ready[slot], 0)) != cudaSuccess) return fail(e);
            // an element's first segment writes its state buffer: the copy out
            // of the element two back must have read it
            if (s == 0 && b >= kSlots &&
                (e = cudaStreamWaitEvent(cs, io->state_done[st], 0)) != cudaSuccess)
                return fail(e);
            // without h0 the first segment starts from zeros; later ones from
            // the state the previous segment left (updated in place)
            const float *seg_h0 = (s == 0 && !hs) ? nullptr : state;
            const gdr_status st_fw = gdr_forward_ex(
                sl + L.q, sl + L.k, sl + L.v, reinterpret_cast<const float *>(sl + L.g),
                reinterpret_cast<const float *>(sl + L.beta), seg_h0, sl + L.out, state, 1, len,
                HK, HV, dk, dv, chunk, cs, qkv_dtype, L.ws_b ? sl + L.ws : nullptr, L.ws_b,
                kSegFlags);
            if (st_fw != GDR_OK) {
                join();
                return st_fw;
            }
            if ((e = cudaEventRecord(io->computed[slot], cs)) != cudaSuccess) return fail(e);
            if ((e = cudaStreamWaitEvent(io->out, io->computed[slot], 0)) != cudaSuccess)
                return fail(e);
            if (len > 0 && (e = cudaMemcpyAsync(ho + row0 * L.tv, sl + L.out, len * L.tv,
                                                cudaMemcpyDeviceToHost, io->out)) != cudaSuccess)
                return fail(e);
            if (s == nseg - 1) {
                if (hh && (e = cudaMemcpyAsync(hh + (size_t)b * sb, state, sb,
                                               cudaMemcpyDeviceToHost, io->out)) != cudaSuccess)
                    return fail(e);
                if ((e = cudaEventRecord(io->state_done[st], io->out)) != cudaSuccess)
                    return fail(e);
            }
            if ((e = cudaEventRecord(io->out_done[slot], io->out)) != cudaSuccess) return fail(e);
        }
    }
    // the caller's stream resumes once every copy out has landed
    if ((e = cudaEventRecord(io->start, io->out)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamWaitEvent(cs, io->start, 0)) != cudaSuccess) return fail(e);
    return GDR_OK;
}

}  // extern "C"
