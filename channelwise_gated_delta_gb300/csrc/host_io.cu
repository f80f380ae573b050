// host_io.cu -- gdr_forward_host: the forward pass on HOST buffers, with the
// host-to-device copies, the compute and the device-to-host copies of
// successive batch elements overlapped.
//
// Batch elements are independent problems, so the batch is streamed through
// two device slots: while element b computes on the caller's stream, the
// inputs of element b + 1 are copied in on a copy-in stream and the outputs
// of element b - 1 are copied out on a copy-out stream.  The link between
// host and device memory is the bound (one direction at a time per copy
// engine; the two directions overlap), so the aim is to keep the copy-in
// stream busy from the first byte to the last.
#include <mutex>
#include <stdint.h>
#include <vector>

#include "common.cuh"
#include "gdr.h"

namespace {

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Per-slot layout: one batch element's inputs, outputs and route workspace.
struct SlotLayout {
    size_t q, k, v, g, beta, h0, out, ht, ws, bytes;   // offsets and total
    size_t q_b, v_b, g_b, beta_b, s_b, ws_b;           // element sizes in bytes
};

SlotLayout slot_layout(int T, int HK, int HV, int dk, int dv, int chunk, int qkv_dtype) {
    SlotLayout L{};
    const size_t es = qkv_dtype == GDR_BF16 ? 2 : 4;
    L.q_b = (size_t)T * HK * dk * es;
    L.v_b = (size_t)T * HV * dv * es;
    L.g_b = (size_t)T * HV * dk * 4;
    L.beta_b = (size_t)T * HV * 4;
    L.s_b = (size_t)HV * dk * dv * 4;
    L.ws_b = gdr_workspace_bytes(1, T, HK, HV, dk, dv, chunk, qkv_dtype, 0);
    size_t off = 0;
    auto put = [&](size_t n) {
        const size_t at = off;
        off = align256(off + n);
        return at;
    };
    L.q = put(L.q_b);
    L.k = put(L.q_b);
    L.v = put(L.v_b);
    L.g = put(L.g_b);
    L.beta = put(L.beta_b);
    L.h0 = put(L.s_b);
    L.out = put(L.v_b);
    L.ht = put(L.s_b);
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
    cudaEvent_t in_ready[kSlots] = {}, computed[kSlots] = {}, out_done[kSlots] = {};
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
        for (int s = 0; s < kSlots && e == cudaSuccess; ++s) {
            e = cudaEventCreateWithFlags(&io.in_ready[s], ef);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&io.computed[s], ef);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&io.out_done[s], ef);
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

}  // namespace

extern "C" {

GDR_API size_t gdr_host_staging_bytes(int B, int T, int HK, int HV, int dk, int dv, int chunk,
                                      int qkv_dtype) {
    if (!valid_shape(B, T, HK, HV, dk, dv, chunk, qkv_dtype) || B == 0) return 0;
    const int slots = B < kSlots ? B : kSlots;
    return slots * slot_layout(T, HK, HV, dk, dv, chunk, qkv_dtype).bytes;
}

GDR_API gdr_status gdr_forward_host(const void *q, const void *k, const void *v, const float *g,
                                    const float *beta, const float *h0, void *out, float *ht,
                                    int B, int T, int HK, int HV, int dk, int dv, int chunk,
                                    void *stream, int qkv_dtype, void *staging,
                                    size_t staging_bytes) {
    if (!valid_shape(B, T, HK, HV, dk, dv, chunk, qkv_dtype)) {
        if (B < 0 || T < 0 || HK <= 0 || HV <= 0 || HV % HK != 0) return GDR_ERR_SHAPE;
        return GDR_ERR_UNSUPPORTED;
    }
    if (B == 0) return GDR_OK;
    if ((long long)T > 0 && (!q || !k || !v || !g || !beta || !out)) return GDR_ERR_NULL;
    const SlotLayout L = slot_layout(T, HK, HV, dk, dv, chunk, qkv_dtype);
    const int slots = B < kSlots ? B : kSlots;
    if (!staging || staging_bytes < (size_t)slots * L.bytes) return GDR_ERR_WORKSPACE;
    if (((uintptr_t)staging & 255u) != 0) return GDR_ERR_ALIGN;

    std::lock_guard<std::mutex> lock(g_io_mutex);
    DeviceIo *io = nullptr;
    cudaError_t e = device_io(&io);
    if (e != cudaSuccess) {
        gdr::record_cuda_error(e);
        return GDR_ERR_CUDA;
    }
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    auto fail = [](cudaError_t err) {
        gdr::record_cuda_error(err);
        return GDR_ERR_CUDA;
    };
    // everything earlier on the caller's stream comes first
    if ((e = cudaEventRecord(io->start, cs)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamWaitEvent(io->in, io->start, 0)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamWaitEvent(io->out, io->start, 0)) != cudaSuccess) return fail(e);

    const char *hq = static_cast<const char *>(q), *hk = static_cast<const char *>(k);
    const char *hv = static_cast<const char *>(v);
    const char *hg = reinterpret_cast<const char *>(g), *hb = reinterpret_cast<const char *>(beta);
    const char *hs = reinterpret_cast<const char *>(h0);
    char *ho = static_cast<char *>(out), *hh = reinterpret_cast<char *>(ht);
    for (int b = 0; b < B; ++b) {
        const int s = b % kSlots;
        char *slot = static_cast<char *>(staging) + (size_t)s * L.bytes;
        // the slot is free once the copies out of its previous element are done
        if (b >= kSlots && (e = cudaStreamWaitEvent(io->in, io->out_done[s], 0)) != cudaSuccess)
            return fail(e);
        struct Copy {
            size_t dst, n;
            const char *src;
        } ins[] = {{L.q, L.q_b, hq + b * L.q_b},       {L.k, L.q_b, hk + b * L.q_b},
                   {L.v, L.v_b, hv + b * L.v_b},       {L.g, L.g_b, hg + b * L.g_b},
                   {L.beta, L.beta_b, hb + b * L.beta_b}, {L.h0, L.s_b, hs ? hs + b * L.s_b : nullptr}};
        for (const Copy &c : ins) {
            if (!c.src || c.n == 0) continue;
            e = cudaMemcpyAsync(slot + c.dst, c.src, c.n, cudaMemcpyHostToDevice, io->in);
            if (e != cudaSuccess) return fail(e);
        }
        if ((e = cudaEventRecord(io->in_ready[s], io->in)) != cudaSuccess) return fail(e);
        if ((e = cudaStreamWaitEvent(cs, io->in_ready[s], 0)) != cudaSuccess) return fail(e);
        const gdr_status st = gdr_forward_ex(
            slot + L.q, slot + L.k, slot + L.v, reinterpret_cast<const float *>(slot + L.g),
            reinterpret_cast<const float *>(slot + L.beta),
            hs ? reinterpret_cast<const float *>(slot + L.h0) : nullptr, slot + L.out,
            hh ? reinterpret_cast<float *>(slot + L.ht) : nullptr, 1, T, HK, HV, dk, dv, chunk,
            cs, qkv_dtype, L.ws_b ? slot + L.ws : nullptr, L.ws_b, 0);
        if (st != GDR_OK) return st;
        if ((e = cudaEventRecord(io->computed[s], cs)) != cudaSuccess) return fail(e);
        if ((e = cudaStreamWaitEvent(io->out, io->computed[s], 0)) != cudaSuccess) return fail(e);
        if (L.v_b && (e = cudaMemcpyAsync(ho + b * L.v_b, slot + L.out, L.v_b,
                                          cudaMemcpyDeviceToHost, io->out)) != cudaSuccess)
            return fail(e);
        if (hh && (e = cudaMemcpyAsync(hh + b * L.s_b, slot + L.ht, L.s_b, cudaMemcpyDeviceToHost,
                                       io->out)) != cudaSuccess)
            return fail(e);
        if ((e = cudaEventRecord(io->out_done[s], io->out)) != cudaSuccess) return fail(e);
    }
    // the caller's stream resumes once every copy out has landed
    if ((e = cudaEventRecord(io->out_done[0], io->out)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamWaitEvent(cs, io->out_done[0], 0)) != cudaSuccess) return fail(e);
    return GDR_OK;
}

}  // extern "C"
