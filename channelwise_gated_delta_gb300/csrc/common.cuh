// common.cuh -- small device helpers shared by the kernels of this library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <vector>
#include <stdint.h>

namespace gdr {

// Element loads/stores for the q/k/v/out dtype.
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Four consecutive elements starting at a 4-element-aligned index, as fp32.
__device__ __forceinline__ float4 load4(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
    uint2 raw = *reinterpret_cast<const uint2 *>(p);
    __nv_bfloat162 lo = *reinterpret_cast<__nv_bfloat162 *>(&raw.x);
    __nv_bfloat162 hi = *reinterpret_cast<__nv_bfloat162 *>(&raw.y);
    float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
    return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void store4(float *p, float4 x) {
    *reinterpret_cast<float4 *>(p) = x;
}
__device__ __forceinline__ void store4(__nv_bfloat16 *p, float4 x) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(x.z, x.w);
    uint2 raw;
    raw.x = *reinterpret_cast<uint32_t *>(&lo);
    raw.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(p) = raw;
}

// Streaming (evict-first) 16-byte global accesses for data touched once.
__device__ __forceinline__ float4 ldg_stream4(const float *p) {
    float4 r;
    asm volatile("ld.global.cs.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
                 : "l"(p));
    return r;
}
__device__ __forceinline__ void stg_stream4(float *p, float4 x) {
    asm volatile("st.global.cs.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(x.x), "f"(x.y),
                 "f"(x.z), "f"(x.w)
                 : "memory");
}

}  // namespace gdr

// Launchers implemented in the .cu files (host side, C++ linkage).
namespace gdr {
// Kernel identities for launch tracing (gdr_trace_enable / gdr_trace_read).
enum KernelId {
    kKernDecode = 0,
    kKernChunkPrep = 1,
    kKernChunkScan = 2,
    kKernFused = 3,
    kKernSegInit = 4,
    kKernSegCombine = 5,
    kKernTree = 6,
    kKernTreePath = 7,
    kKernTreeGram = 8,
    kKernTreeSolve = 9,
    kKernChunkScanTc = 10,
    kKernChunkPrepTc = 11,
    kNumKernels = 12
};
// Called by the launchers around each launch; no-ops unless tracing is on.
void trace_begin(int kernel, cudaStream_t stream);
void trace_end(int kernel, cudaStream_t stream);

struct Problem {
    const void *q, *k, *v;
    const float *g, *beta, *h0;
    void *out;
    float *ht;
    int B, T, HK, HV, dk, dv, chunk;
    int bf16;      // 1: q/k/v/out are bfloat16, 0: float32
    int g_scalar;  // 1: g is [rows][HV] (one log-decay per token and value head), 0: [rows][HV][dk]
};

cudaError_t launch_decode(const Problem &p, cudaStream_t stream);
bool tc_prefill_supported(const Problem &p);
// api.cu: device address of the library's error word on the current device,
// and a setter for gdr_last_cuda_error().
cudaError_t device_error_word(int **out);
int record_cuda_error(cudaError_t e);
cudaError_t launch_tc_prefill(const Problem &p, int *dev_error, cudaStream_t stream);
size_t generic_prefill_workspace_bytes(const Problem &p);
// tc_scan: the state scan on the tensor cores (launch_chunk_scan_tc) rather
// than on CUDA cores; the prep writes its records for it.  segments >= 2
// (tc_scan only): that scan cut into segments (scan_segment_count), with
// the workspace generic_prefill_workspace_bytes(p, segments).
size_t generic_prefill_workspace_bytes(const Problem &p, int segments);
cudaError_t launch_generic_prefill(const Problem &p, void *workspace, cudaStream_t stream,
                                   bool tc_scan = false, int segments = 0);

// Packed variable-length batches (p.B = number of entries in the table, the
// pointers those of the packed tensors).
// Decode of single tokens: rows[b] = {token row, state slot}.
cudaError_t launch_decode_rows(const Problem &p, const int2 *rows, cudaStream_t stream);
// Tensor-core prefill: seqs[s] = {first token row, length, state slot, -};
// seq_maps: one tensor-map set per sequence (tc_seq_maps_bytes() each,
// 64-byte aligned, in device memory), filled on the host by tc_encode_seq_maps.
// A non-null v_row (o_row) replaces the sequence's values (outputs) by a
// one-row [1][HV][128] bf16 device tensor: the values read as zeros past its
// row 0 (zero-filled loads), the outputs past row 0 are dropped.
size_t tc_seq_maps_bytes();
cudaError_t tc_encode_seq_maps(const Problem &p, size_t tok0, int L, void *dst,
                               const void *v_row = nullptr, void *o_row = nullptr);
cudaError_t launch_tc_prefill_varlen(const Problem &p, const void *seq_maps, const int4 *seqs,
                                     int nseq, int *dev_error, cudaStream_t stream);
// seqs[s].w of that launch: the state the sequence starts from (0: its h0
// slot; kSeqStartZero: zero; kSeqStartIdentity: the identity, dk = dv).
constexpr int kSeqStartZero = 1;
constexpr int kSeqStartIdentity = 2;
// CUDA-core chunked prefill: chunks[i] = {first token row, length} of every
// sequence's chunks, seqs[s] = {first token row, length, state slot, index
// of its first chunk}; records: generic_varlen_record_bytes(p, nchunks).
size_t generic_varlen_record_bytes(const Problem &p, long long nchunks);
// tc_scan: also nseg sequences cut into seg_P segments (seg_seqs on the
// host, records addressed as packed chunks), workspace seg_ws of
// scan_segmented_bytes(p, nseg, seg_P); p.B counts the whole ones only.
struct ScanSeq;
cudaError_t launch_generic_prefill_varlen(const Problem &p, void *records, const int2 *chunks,
                                          int nchunks, const int4 *seqs, cudaStream_t stream,
                                          bool tc_scan = false, const ScanSeq *seg_seqs = nullptr,
                                          int nseg = 0, int seg_P = 0, void *seg_ws = nullptr);
// The state scan of the chunked prefill on the tensor cores (scan_tc.cu):
// records in the tensor-core layout written by the prep kernel, rec_floats
// floats each; dense batches (seqs == nullptr) or nseq packed sequences.
bool scan_tc_supported(const Problem &p);
cudaError_t launch_chunk_scan_tc(const Problem &p, const float *records, size_t rec_floats,
                                 const int4 *seqs, int nseq, cudaStream_t stream);
// The chunk prep of that route on the tensor cores (prep_tc.cu; dk = dv =
// 128, chunk 64): the same records as gdr_chunk_prep's tensor-core layout,
// rec_floats floats each; dense batches (chunks == nullptr) or the nchunks
// chunks {first row, length} of a packed batch.
bool prep_tc_supported(const Problem &p);
cudaError_t launch_chunk_prep_tc(const Problem &p, float *records, size_t rec_floats,
                                 const int2 *chunks, int nchunks, cudaStream_t stream);
// One run of that scan in a segmented launch: tokens tok0 .. tok0 + T - 1,
// whose chunk c of value head hv has its record at rec_base + hv * hv_stride
// + c * c_stride; the state starts from slot `slot` of p.h0 and ends in slot
// `slot` of p.ht.  kRunZeroValues: the values read as zero (the run from
// the identity then ends in the segment's map M); kRunNoOutputs: the
// outputs are dropped; kRunStartZero / kRunStartIdentity: the state starts
// at zero / the identity instead of slot `slot` of p.h0.
struct ScanRun {
    long long tok0, rec_base;
    int T, slot, hv_stride, c_stride, flags, pad;
};
constexpr int kRunZeroValues = 1;
constexpr int kRunNoOutputs = 2;
constexpr int kRunStartZero = 4;      // the state starts at zero (h0 not read)
constexpr int kRunStartIdentity = 8;  // the state starts at the identity (dk = dv)
cudaError_t launch_chunk_scan_runs(const Problem &p, const float *records, size_t rec_floats,
                                   const ScanRun *runs, int nrun, cudaStream_t stream);
// Tree verification on CUDA cores: p.B trees of p.T <= p.chunk tokens each,
// parents [B][T] (device); records: generic_tree_record_bytes(p).
size_t generic_tree_record_bytes(const Problem &p);
// Tree verification on the tensor cores (tc_prefill_supported, T <= 64):
// parents [B][T] on the device.
cudaError_t launch_tc_tree(const Problem &p, const int *parents, int *dev_error,
                           cudaStream_t stream);
cudaError_t launch_generic_tree(const Problem &p, void *records, const int *parents,
                                cudaStream_t stream);
// Tree verification of up to 512 tokens as one blocked unit-lower solve
// (tree_blocked.cu): parents [B][T] on the device, workspace
// tree_blocked_workspace_bytes(p), 256-byte aligned.  variant:
// kTreeGramPerValueHead keeps a scalar gate's gram per value head (the
// fused form) instead of once per key head.
constexpr unsigned kTreeGramPerValueHead = 1u;
bool tree_blocked_supported(const Problem &p);
size_t tree_blocked_workspace_bytes(const Problem &p);
cudaError_t launch_tree_blocked(const Problem &p, void *workspace, const int *parents,
                                unsigned variant, cudaStream_t stream);

// Chunk-parallel state scan on the tensor-core route (segments.cu): the
// segment count chosen for `p` (0: not segmented) under `flags`, its
// workspace, and the launches.
int segment_count(const Problem &p, unsigned flags);
size_t segmented_workspace_bytes(const Problem &p, int segments);
cudaError_t launch_segmented_prefill(const Problem &p, int segments, void *workspace,
                                     int *dev_error, cudaStream_t stream);
// The segments a sequence of T tokens is cut into when P are asked for: P
// segments of ceil(chunks / P) whole chunks (64 tokens each unless `chunk`
// says otherwise), the last possibly
// shorter, so fewer than P when the chunks do not spread that far; 0 when
// fewer than two.
inline int effective_segments(int T, int P, int chunk = 64) {
    const int nch = (T + chunk - 1) / chunk;
    if (P < 2 || nch < 2) return 0;
    const int per = (nch + P - 1) / P;
    const int eff = (nch + per - 1) / per;
    return eff >= 2 ? eff : 0;
}
// Packed batches: one sequence of a segmented launch (first token row,
// length, index of its h0 / ht slot).
struct SegSeq {
    size_t row0;
    int T;
    int slot;
};
// The segment count for a packed batch whose tensor-core prefill sequences
// have `lengths` (0: none cut); (*cut)[i] marks the sequences cut into that
// many segments, the rest walk whole.
int varlen_segment_count(const Problem &p, const int *lengths, int n, unsigned flags,
                         std::vector<char> *cut);
size_t segmented_list_workspace_bytes(const Problem &p, int nseq, int P);
cudaError_t launch_segmented_list(const Problem &p, const SegSeq *seqs, int nseq, int P,
                                  void *workspace, int *dev_error, cudaStream_t stream);
// The same segmented scan on the route of chunk records (the CUDA-core prep,
// then the tensor-core state scan; dk = dv = 128): the segment count for a
// dense batch under `flags` (0: not segmented), and for packed sequences of
// `lengths` with (*cut)[i] marking those cut; the workspace after the
// records; the launches, given every sequence's first token row, length,
// state slot and record addressing (rec_base: its chunk 0 of value head 0).
struct ScanSeq {
    long long tok0, rec_base;
    int T, slot, hv_stride, c_stride;
};
int scan_segment_count(const Problem &p, unsigned flags);
int scan_varlen_segment_count(const Problem &p, const int *lengths, int n, unsigned flags,
                              std::vector<char> *cut);
size_t scan_segmented_bytes(const Problem &p, int nseq, int P);
cudaError_t launch_scan_segmented(const Problem &p, const float *records, size_t rec_floats,
                                  const ScanSeq *seqs, int nseq, int P, void *workspace,
                                  cudaStream_t stream);
}  // namespace gdr
