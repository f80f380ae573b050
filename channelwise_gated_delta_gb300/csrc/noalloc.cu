// noalloc.cu -- gdr_forward_chunked_noalloc: the chunked CUDA-core prefill
// with its scratch in a fixed device array, for callers that cannot allocate
// device memory.
//
// Who needs it: code that runs where cudaMalloc is not allowed or not
// acceptable -- an embedding runtime whose memory planner owns every device
// byte up front and hands operators only their inputs and outputs (so no
// operator may allocate on its own), a latency-critical serving loop that
// must never hit cudaMalloc's implicit device-wide synchronisation, or a
// plugin inside a host process whose caching allocator must remain the only
// owner of device memory.  Such callers can still pass inputs and outputs;
// they just cannot provide or obtain the workspace the chunked prefill needs.
//
// The scratch is a file-scope __device__ array of GDR_NOALLOC_SCRATCH_BYTES
// bytes.  Every GPU that loads this library holds it until the process exits.
// In host code the array's name is only a host-side stand-in for the symbol,
// so the device address is obtained with cudaGetSymbolAddress, once per
// device, on the first call made with that device current, and cached.
#include <mutex>
#include <vector>

#include "common.cuh"
#include "gdr.h"

static __device__ __align__(256) unsigned char g_noalloc_scratch[GDR_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_noalloc_mutex;
std::vector<void *> g_noalloc_addr;  // per device ordinal; nullptr until set up

// Device address of g_noalloc_scratch on the current device (set-up on first use).
cudaError_t noalloc_scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if ((int)g_noalloc_addr.size() <= dev) g_noalloc_addr.resize(dev + 1, nullptr);
    if (!g_noalloc_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" GDR_API gdr_status gdr_forward_chunked_noalloc(
    const void *q, const void *k, const void *v, const float *g, const float *beta,
    const float *h0, void *out, float *ht, int B, int T, int HK, int HV, int dk, int dv,
    int chunk, void *stream, int qkv_dtype) {
    const unsigned flags = GDR_FLAG_FORCE_CHUNKED | GDR_FLAG_FORCE_GENERIC;
    // Reject problems whose scratch would not fit before touching the GPU.
    // (gdr_workspace_bytes returns 0 for invalid shapes; gdr_forward_ex then
    // reports the precise argument error.)
    const size_t need = gdr_workspace_bytes(B, T, HK, HV, dk, dv, chunk, qkv_dtype, flags);
    if (need > (size_t)GDR_NOALLOC_SCRATCH_BYTES) return GDR_ERR_WORKSPACE;
    void *scratch = nullptr;
    const cudaError_t e = noalloc_scratch_address(&scratch);
    if (e != cudaSuccess) {
        gdr::record_cuda_error(e);
        return GDR_ERR_CUDA;
    }
    // The chunked prefill writes every scratch word it later reads, within
    // the call, so the previous call's leftovers need no clearing.
    return gdr_forward_ex(q, k, v, g, beta, h0, out, ht, B, T, HK, HV, dk, dv, chunk, stream,
                          qkv_dtype, scratch, (size_t)GDR_NOALLOC_SCRATCH_BYTES, flags);
}
