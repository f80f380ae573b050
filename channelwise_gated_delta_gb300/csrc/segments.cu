// segments.cu -- the chunk-parallel state scan on the tensor-core prefill.
//
// The chunk-to-chunk state carry of the chunkwise form (page "Reorder
// channelwise gated delta rule chunked hot loops for autovectorization",
// pytorch/executorch PR #21021, second commit summary) is serial: one CTA
// walks a head's chunks in order.  When batch x heads leaves most SMs idle,
// the sequence is cut into P segments of whole chunks.  Over a segment the
// recurrence is an affine map of the state, S_end = M S_start + c, with M
// [dk][dk] depending on k, g and beta only: M is the end state of a run from
// S_start = I with v = 0, c the end state of a run from S_start = 0.
//
//   wave A  (one launch, all concurrent)  segment 0 from h0 -> S_1;
//           for p = 1 .. P-2: the runs that give M_p and c_p
//   combine S_{p+1} = M_p S_p + c_p, p = 1 .. P-2 (gdr_segment_combine)
//   wave B  (one launch) segment p = 1 .. P-1 from S_p: outputs, and ht
//
// Both waves are the packed-sequence tensor-core kernel: every run is one
// "sequence" with its own tensor maps and state slot.  The map runs read
// their values from a one-row zero tensor (each row past row 0 is the loads'
// zero fill) and send their outputs to a one-row scratch tensor (each row
// past row 0 falls outside it and is dropped), so they move no value or
// output bytes.  The critical path is two segments instead of P.
//
// State slots, a group of 2P-3 per batch element b (each slot HV x [128][128]
// f32): X_1, M_1, X_2, M_2, X_3, ..., M_{P-2}, X_{P-1} -- X_p at 2(p-1), M_p
// at 2p-1.  X_1 takes a copy of h0[b] when there is one; the map runs start
// from the identity and the c runs from zero by their run flags, so no slot
// needs filling.  Wave A leaves X_1 = S_1, M_p and X_{p+1} = c_p; the
// combine turns X_{p+1} into S_{p+1} in place; wave B runs segment p in place
// on X_p, which leaves the final state in X_{P-1}.
#include <algorithm>
#include <mutex>
#include <string.h>
#include <vector>

#include "common.cuh"
#include "gdr.h"

namespace gdr {
namespace {

constexpr int kD = 128;   // dk = dv of the tensor-core route
constexpr int kC = 64;    // its chunk
constexpr size_t kSlotFloats = (size_t)kD * kD;
// Shortest segment the automatic choice makes, in chunks: below this the
// per-launch fill and the combine cost more than the shorter walk saves.
constexpr int kMinSegmentChunks = 8;
constexpr int kCombineThreads = 256;
constexpr int kMtLd = kD + 4;  // transposed M rows, padded (16-byte aligned)

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// A zero value row for the map runs: device memory that is zero at module
// load and never written, so no call has to clear it (HV x 128 bf16 of it
// at most; a larger HV clears a row of the workspace instead).
constexpr size_t kZeroRowBytes = 1u << 20;
__device__ __align__(256) unsigned char g_zero_row[kZeroRowBytes];

// Its device address on the current device (looked up once per device).
cudaError_t zero_row_address(void **out) {
    static std::mutex mu;
    static std::vector<void *> cache;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if ((int)cache.size() <= dev) cache.resize(dev + 1, nullptr);
    if (!cache[dev]) {
        void *p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_zero_row)) != cudaSuccess) return e;
        cache[dev] = p;
    }
    *out = cache[dev];
    return cudaSuccess;
}

// SM count of the current device, looked up once per device; 0 if unknown.
int sm_count() {
    static std::mutex mu;
    static std::vector<int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    if ((int)cache.size() <= dev) cache.resize(dev + 1, -1);
    if (cache[dev] < 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        cache[dev] = n;
    }
    return cache[dev];
}

struct Segments {
    int P = 0;        // number of segments
    int group = 0;    // state slots per sequence, 2P - 3 (1 when P = 2)
    int nseq = 0;     // sequences
    int nA = 0, nB = 0;                // runs in wave A and wave B
    size_t off_seqA = 0, off_mapA = 0, off_seqB = 0, off_mapB = 0;
    size_t off_zero = 0, off_scratch = 0, off_state = 0, table_bytes = 0, total = 0;
};

// Workspace of nseq sequences cut into P segments each: the tables (both
// waves' run records and tensor maps), a zero value row (used when HV is
// past the static one), the scratch output row and 2P - 3 state slots per
// sequence.
Segments plan_seqs(const Problem &p, int nseq, int P) {
    Segments s;
    if (P < 2 || nseq <= 0) return s;
    s.P = P;
    s.nseq = nseq;
    s.group = 2 * s.P - 3;
    s.nA = nseq * s.group;
    s.nB = nseq * (s.P - 1);
    const size_t maps = tc_seq_maps_bytes();
    size_t off = 0;
    s.off_seqA = off;
    off = align256(off + (size_t)s.nA * sizeof(int4));
    s.off_mapA = off;
    off = align256(off + (size_t)s.nA * maps);
    s.off_seqB = off;
    off = align256(off + (size_t)s.nB * sizeof(int4));
    s.off_mapB = off;
    off = align256(off + (size_t)s.nB * maps);
    s.table_bytes = off;
    const size_t row = (size_t)p.HV * kD * 2;  // one bf16 token row of v / o
    s.off_zero = off;
    off = align256(off + row);
    s.off_scratch = off;
    off = align256(off + row);
    s.off_state = off;
    off += (size_t)s.nA * p.HV * kSlotFloats * sizeof(float);
    s.total = off;
    return s;
}

// A dense batch: every batch element is one sequence of p.T tokens.
Segments plan(const Problem &p, int P) {
    const int eff = effective_segments(p.T, P);
    return eff >= 2 ? plan_seqs(p, p.B, eff) : Segments{};
}

// S_{p+1} = M_p S_p + c_p for p = 1 .. P-2, in place on the X slots.  One
// CTA per (b, hv, SLAB-column slab of the state): the columns of the state
// are independent, so the slab walks the whole chain alone, kept in shared
// memory between steps.  M_p is staged transposed (Mt[k][r]) so that a
// thread's R = SLAB / 8 rows at one k are one vector load; each thread owns
// an R x 4 tile (rows R rg .., columns 4 cg .. of the slab).  f32 FMAs, k in
// order.  SLAB = 16 (eight CTAs per head) when that many CTAs fit on the
// SMs at once, else 32.
template <int SLAB>
__global__ void __launch_bounds__(kCombineThreads) gdr_segment_combine(float *__restrict__ state,
                                                                       int HV, int P) {
    constexpr int R = SLAB / 8, CG = SLAB / 4, NS = kD / SLAB;
    static_assert(R * 4 * kCombineThreads == kD * SLAB, "one R x 4 tile per thread");
    extern __shared__ float smc[];
    float *Mt = smc;                 // [128][kMtLd]
    float *Xs = smc + kD * kMtLd;    // [128][SLAB]
    const int slab = blockIdx.x % NS, head = blockIdx.x / NS;
    const int hv = head % HV, b = head / HV;
    const int group = 2 * P - 3;
    auto slot = [&](int j) { return state + ((size_t)(b * group + j) * HV + hv) * kSlotFloats; };
    const int tid = threadIdx.x;
    const int c0 = SLAB * slab;
    const int cg = tid % CG, rg = tid / CG;
    constexpr int kXLoads = kD * SLAB / 4 / kCombineThreads;

    {
        const float *x1 = slot(0);
        float4 x[kXLoads];
#pragma unroll
        for (int u = 0; u < kXLoads; ++u) {
            const int i = tid + u * kCombineThreads, r = i / CG, qd = i % CG;
            x[u] = *reinterpret_cast<const float4 *>(x1 + (size_t)r * kD + c0 + 4 * qd);
        }
#pragma unroll
        for (int u = 0; u < kXLoads; ++u) {
            const int i = tid + u * kCombineThreads, r = i / CG, qd = i % CG;
            *reinterpret_cast<float4 *>(Xs + r * SLAB + 4 * qd) = x[u];
        }
    }
    for (int p = 1; p <= P - 2; ++p) {
        const float *M = slot(2 * p - 1);
        float *X = slot(2 * p);  // c_p in, S_{p+1} out
        // this thread's c_p tile and M_p share, all loads in flight at once
        float4 cv[R];
#pragma unroll
        for (int e = 0; e < R; ++e)
            cv[e] = *reinterpret_cast<const float4 *>(X + (size_t)(R * rg + e) * kD + c0 + 4 * cg);
        constexpr int kMLoads = kD * (kD / 4) / kCombineThreads;
        float4 m[kMLoads];
#pragma unroll
        for (int u = 0; u < kMLoads; ++u) {
            // lanes take consecutive rows, so the transposed stores use all banks
            const int i = tid + u * kCombineThreads;
            const int r = (i & 31) + 32 * (i >> 10), kq = (i >> 5) & 31;
            m[u] = *reinterpret_cast<const float4 *>(M + (size_t)r * kD + 4 * kq);
        }
        __syncthreads();  // Xs written; the previous step's reads of Mt done
#pragma unroll
        for (int u = 0; u < kMLoads; ++u) {
            const int i = tid + u * kCombineThreads;
            const int r = (i & 31) + 32 * (i >> 10), kq = (i >> 5) & 31;
            Mt[(4 * kq + 0) * kMtLd + r] = m[u].x;
            Mt[(4 * kq + 1) * kMtLd + r] = m[u].y;
            Mt[(4 * kq + 2) * kMtLd + r] = m[u].z;
            Mt[(4 * kq + 3) * kMtLd + r] = m[u].w;
        }
        __syncthreads();
        float acc[R][4] = {};
#pragma unroll 8
        for (int k = 0; k < kD; ++k) {
            float mv[R];
            if constexpr (R == 4) {
                const float4 mk = *reinterpret_cast<const float4 *>(Mt + k * kMtLd + R * rg);
                mv[0] = mk.x, mv[1] = mk.y, mv[2] = mk.z, mv[3] = mk.w;
            } else {
                const float2 mk = *reinterpret_cast<const float2 *>(Mt + k * kMtLd + R * rg);
                mv[0] = mk.x, mv[1] = mk.y;
            }
            const float4 x = *reinterpret_cast<const float4 *>(Xs + k * SLAB + 4 * cg);
            const float xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int e = 0; e < R; ++e)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) acc[e][jj] = fmaf(mv[e], xv[jj], acc[e][jj]);
        }
        __syncthreads();  // every read of Xs done before it is overwritten
#pragma unroll
        for (int e = 0; e < R; ++e) {
            const int r = R * rg + e;
            const float4 c = cv[e];
            const float4 y = make_float4(acc[e][0] + c.x, acc[e][1] + c.y, acc[e][2] + c.z,
                                         acc[e][3] + c.w);
            *reinterpret_cast<float4 *>(X + (size_t)r * kD + c0 + 4 * cg) = y;
            *reinterpret_cast<float4 *>(Xs + r * SLAB + 4 * cg) = y;
        }
    }
}

constexpr size_t combine_smem(int slab) {
    return ((size_t)kD * kMtLd + (size_t)kD * slab) * sizeof(float);
}

// The combine over nseq groups of 2P - 3 slots (nothing to chain when P = 2).
cudaError_t launch_combine(const Problem &p, float *state, int nseq, int P, cudaStream_t stream) {
    if (P < 3) return cudaSuccess;
    const int sms = sm_count();
    const bool narrow = sms > 0 && (long long)nseq * p.HV * (kD / 16) <= sms;
    auto combine = [&](auto kernel, int slab) -> cudaError_t {
        cudaError_t r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)combine_smem(slab));
        if (r != cudaSuccess) return r;
        trace_begin(kKernSegCombine, stream);
        kernel<<<(unsigned)(nseq * p.HV * (kD / slab)), kCombineThreads, combine_smem(slab),
                 stream>>>(state, p.HV, P);
        trace_end(kKernSegCombine, stream);
        return cudaGetLastError();
    };
    return narrow ? combine(gdr_segment_combine<16>, 16) : combine(gdr_segment_combine<32>, 32);
}

// X_{P-1} of every sequence into its ht slot (slots[b]): one strided copy
// when the slots are the sequences' order, else one copy per sequence.
cudaError_t copy_final_states(const Problem &p, const float *state, const std::vector<int> &slots,
                              int P, cudaStream_t stream) {
    if (!p.ht) return cudaSuccess;
    const int nseq = (int)slots.size(), group = 2 * P - 3;
    const size_t head_bytes = (size_t)p.HV * kSlotFloats * sizeof(float);
    const float *last = state + (size_t)2 * (P - 2) * p.HV * kSlotFloats;
    bool in_order = true;
    for (int b = 0; b < nseq; ++b) in_order = in_order && slots[b] == b;
    if (in_order)
        return cudaMemcpy2DAsync(p.ht, head_bytes, last, (size_t)group * head_bytes, head_bytes,
                                 nseq, cudaMemcpyDeviceToDevice, stream);
    cudaError_t e = cudaSuccess;
    for (int b = 0; b < nseq && e == cudaSuccess; ++b)
        e = cudaMemcpyAsync(p.ht + (size_t)slots[b] * p.HV * kSlotFloats,
                            last + (size_t)b * group * p.HV * kSlotFloats, head_bytes,
                            cudaMemcpyDeviceToDevice, stream);
    return e;
}

// h0 of every sequence (slots[b]) into its X_1 slot: one strided copy when
// the slots are the sequences' order, else one copy per sequence.
cudaError_t copy_initial_states(const Problem &p, float *state, const std::vector<int> &slots,
                                int P, cudaStream_t stream) {
    if (!p.h0) return cudaSuccess;
    const int nseq = (int)slots.size(), group = 2 * P - 3;
    const size_t head_bytes = (size_t)p.HV * kSlotFloats * sizeof(float);
    bool in_order = true;
    for (int b = 0; b < nseq; ++b) in_order = in_order && slots[b] == b;
    if (in_order)
        return cudaMemcpy2DAsync(state, (size_t)group * head_bytes, p.h0, head_bytes, head_bytes,
                                 nseq, cudaMemcpyDeviceToDevice, stream);
    cudaError_t e = cudaSuccess;
    for (int b = 0; b < nseq && e == cudaSuccess; ++b)
        e = cudaMemcpyAsync(state + (size_t)b * group * p.HV * kSlotFloats,
                            p.h0 + (size_t)slots[b] * p.HV * kSlotFloats, head_bytes,
                            cudaMemcpyDeviceToDevice, stream);
    return e;
}

// Which of n sequences of `lengths` (chunks of `chunk` tokens) to cut, and
// into how many segments: forced (flags' segment count), every sequence that
// spreads over exactly that many; automatic, the largest q >= 3 for which
// every sequence's CTA and wave A's 2q - 3 runs per cut sequence fit on the
// SMs in one wave, cutting the sequences of kMinSegmentChunks q chunks or
// more that spread over exactly q.  0: none cut.
int choose_list_segments(const Problem &p, const int *lengths, int n, unsigned flags, int chunk,
                         std::vector<char> *cut) {
    auto select = [&](int P, int min_chunks) {
        int m = 0;
        for (int i = 0; i < n; ++i) {
            const int nch = (lengths[i] + chunk - 1) / chunk;
            (*cut)[i] = nch >= min_chunks && effective_segments(lengths[i], P, chunk) == P;
            m += (*cut)[i];
        }
        return m;
    };
    const int forced = (int)((flags >> 8) & 0xffu);
    int P = 0;
    if (forced) {
        P = forced;
        if (select(P, 2) == 0) P = 0;
    } else {
        const int sms = sm_count();
        if (sms <= 0) return 0;
        int longest = 0;
        for (int i = 0; i < n; ++i) longest = std::max(longest, lengths[i]);
        for (int q = ((longest + chunk - 1) / chunk) / kMinSegmentChunks; q >= 3 && !P; --q) {
            const int m = select(q, q * kMinSegmentChunks);
            if (m > 0 && (long long)p.HV * ((long long)(2 * q - 3) * m + (n - m)) <= sms) P = q;
        }
    }
    if (P == 0) {
        cut->assign((size_t)n, 0);
        return 0;
    }
    long long m = 0;
    for (char c : *cut) m += c;
    if (m * (2 * P - 3) * p.HV * 4 > 0x7fffffffLL) {
        cut->assign((size_t)n, 0);
        return 0;
    }
    return P;
}

// The dense-batch count: wave A runs B HV (2P - 3) CTAs, one per SM; the
// largest P that keeps it to one wave, with segments of kMinSegmentChunks
// chunks or more; forced counts as asked (fewer when the chunks do not
// spread that far).
int dense_segments(const Problem &p, unsigned flags, int chunk) {
    const int nch = (p.T + chunk - 1) / chunk;
    const int forced = (int)((flags >> 8) & 0xffu);
    int P = forced;
    if (!forced) {
        const int sms = sm_count();
        const long long units = (long long)p.B * p.HV;
        if (sms <= 0 || units <= 0) return 0;
        P = (int)((sms / units + 3) / 2);
        P = std::min(P, nch / kMinSegmentChunks);
        if (P < 3) return 0;  // two segments walk as long as one
    }
    const int eff = effective_segments(p.T, P, chunk);
    if (eff < 2 || (!forced && eff < 3)) return 0;
    // every grid (4 blocks per slot and head at most) and slot index in int
    if ((long long)p.B * (2 * eff - 3) * p.HV * 4 > 0x7fffffffLL) return 0;
    return eff;
}

}  // namespace

int segment_count(const Problem &p, unsigned flags) {
    if (flags & GDR_FLAG_NO_SEGMENTS) return 0;
    if (!tc_prefill_supported(p) || p.B <= 0 || p.T < 2) return 0;
    return dense_segments(p, flags, kC);
}

size_t segmented_workspace_bytes(const Problem &p, int segments) {
    return plan(p, segments).total;
}

int varlen_segment_count(const Problem &p, const int *lengths, int n, unsigned flags,
                         std::vector<char> *cut) {
    cut->assign((size_t)std::max(n, 0), 0);
    if ((flags & GDR_FLAG_NO_SEGMENTS) || n <= 0) return 0;
    Problem one = p;
    one.B = 1;
    one.T = 2;
    if (!tc_prefill_supported(one)) return 0;
    return choose_list_segments(p, lengths, n, flags, kC, cut);
}

size_t segmented_list_workspace_bytes(const Problem &p, int nseq, int P) {
    return plan_seqs(p, nseq, P).total;
}

cudaError_t launch_segmented_list(const Problem &p, const SegSeq *seqs, int nseq, int P,
                                  void *workspace, int *dev_error, cudaStream_t stream) {
    const Segments s = plan_seqs(p, nseq, P);
    if (s.P != P || s.total == 0) return cudaErrorInvalidValue;
    for (int i = 0; i < nseq; ++i)
        if (effective_segments(seqs[i].T, P) != P) return cudaErrorInvalidValue;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    const size_t row_bytes = (size_t)p.HV * kD * 2;
    void *zero_row = nullptr;
    cudaError_t e = cudaSuccess;
    if (row_bytes <= kZeroRowBytes) {
        if ((e = zero_row_address(&zero_row)) != cudaSuccess) return e;
    } else {
        zero_row = ws + s.off_zero;  // cleared below
    }
    void *scratch_row = ws + s.off_scratch;
    float *state = reinterpret_cast<float *>(ws + s.off_state);
    const size_t maps = tc_seq_maps_bytes();

    // tables: per run {first token row, length, state slot, start flag} and
    // its tensor maps
    std::vector<unsigned char> host(s.table_bytes, 0);
    int4 *seqA = reinterpret_cast<int4 *>(host.data() + s.off_seqA);
    int4 *seqB = reinterpret_cast<int4 *>(host.data() + s.off_seqB);
    int a = 0, bb = 0;
    for (int b = 0; b < nseq; ++b) {
        const SegSeq &sq = seqs[b];
        const int base = b * s.group;
        const int seg_len = ((sq.T + kC - 1) / kC + P - 1) / P * kC;  // whole chunks
        auto seg_t0 = [&](int q) { return q * seg_len; };
        auto seg_len_of = [&](int q) { return std::min(sq.T, (q + 1) * seg_len) - q * seg_len; };
        auto add = [&](int4 *tab, size_t off_map, int &n, int q, int slot_j, const void *v_row,
                       void *o_row, int start) {
            const size_t tok0 = sq.row0 + seg_t0(q);
            tab[n] = make_int4((int)tok0, seg_len_of(q), base + slot_j, start);
            const cudaError_t r = tc_encode_seq_maps(p, tok0, seg_len_of(q),
                                                     host.data() + off_map + (size_t)n * maps,
                                                     v_row, o_row);
            ++n;
            return r;
        };
        e = add(seqA, s.off_mapA, a, 0, 0, nullptr, nullptr, p.h0 ? 0 : kSeqStartZero);
        for (int q = 1; q <= s.P - 2 && e == cudaSuccess; ++q) {
            e = add(seqA, s.off_mapA, a, q, 2 * q - 1, zero_row, scratch_row, kSeqStartIdentity);  // M_q
            if (e == cudaSuccess)
                e = add(seqA, s.off_mapA, a, q, 2 * q, nullptr, scratch_row, kSeqStartZero);  // c_q
        }
        for (int q = 1; q <= s.P - 1 && e == cudaSuccess; ++q)
            e = add(seqB, s.off_mapB, bb, q, 2 * (q - 1), nullptr, nullptr, 0);
        if (e != cudaSuccess) return e;
    }
    // pageable source: the call returns once the bytes have been taken
    e = cudaMemcpyAsync(ws, host.data(), s.table_bytes, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;

    // h0 into the X_1 slots (and, past the static zero row's size, a zero
    // row of the workspace for the map runs)
    std::vector<int> seq_slots((size_t)nseq);
    for (int b = 0; b < nseq; ++b) seq_slots[b] = seqs[b].slot;
    if (zero_row == ws + s.off_zero && (e = cudaMemsetAsync(zero_row, 0, row_bytes, stream)) != cudaSuccess)
        return e;
    e = copy_initial_states(p, state, seq_slots, s.P, stream);
    if (e != cudaSuccess) return e;

    Problem wave = p;
    wave.h0 = state;
    wave.ht = state;
    wave.T = 0;
    wave.B = s.nA;
    e = launch_tc_prefill_varlen(wave, ws + s.off_mapA,
                                 reinterpret_cast<const int4 *>(ws + s.off_seqA), s.nA, dev_error,
                                 stream);
    if (e != cudaSuccess) return e;
    e = launch_combine(p, state, nseq, s.P, stream);
    if (e != cudaSuccess) return e;
    wave.B = s.nB;
    e = launch_tc_prefill_varlen(wave, ws + s.off_mapB,
                                 reinterpret_cast<const int4 *>(ws + s.off_seqB), s.nB, dev_error,
                                 stream);
    if (e != cudaSuccess) return e;
    return copy_final_states(p, state, seq_slots, s.P, stream);
}

cudaError_t launch_segmented_prefill(const Problem &p, int segments, void *workspace,
                                     int *dev_error, cudaStream_t stream) {
    const Segments s = plan(p, segments);
    if (s.P != segments || s.total == 0) return cudaErrorInvalidValue;
    std::vector<SegSeq> seqs((size_t)p.B);
    for (int b = 0; b < p.B; ++b) seqs[b] = SegSeq{(size_t)b * p.T, p.T, b};
    return launch_segmented_list(p, seqs.data(), p.B, segments, workspace, dev_error, stream);
}


// ---- the route of chunk records (CUDA-core prep, tensor-core state scan)
//
// Same waves, slots and combine as above; the runs are scan CTAs over the
// records the prep kernel wrote for every chunk at once, so a run only
// needs its first record, its length and its flags: a map run reads the
// values as zero (kRunZeroValues) and, like a c run, drops its outputs
// (kRunNoOutputs).  Segments are whole chunks of p.chunk tokens.

namespace {

struct ScanSegments {
    int P = 0, group = 0, nseq = 0, nA = 0, nB = 0;
    size_t off_runA = 0, off_runB = 0, table_bytes = 0, off_state = 0, total = 0;
};

ScanSegments plan_scan(const Problem &p, int nseq, int P) {
    ScanSegments s;
    if (P < 2 || nseq <= 0) return s;
    s.P = P;
    s.nseq = nseq;
    s.group = 2 * P - 3;
    s.nA = nseq * s.group;
    s.nB = nseq * (P - 1);
    size_t off = 0;
    s.off_runA = off;
    off = align256(off + (size_t)s.nA * sizeof(ScanRun));
    s.off_runB = off;
    off = align256(off + (size_t)s.nB * sizeof(ScanRun));
    s.table_bytes = off;
    s.off_state = off;
    off += (size_t)s.nA * p.HV * kSlotFloats * sizeof(float);
    s.total = off;
    return s;
}

// dk = dv = 128 (the combine's state), the tensor-core scan, not forced
// onto the CUDA-core kernels
bool scan_segmentable(const Problem &p, unsigned flags) {
    return !(flags & (GDR_FLAG_NO_SEGMENTS | GDR_FLAG_FORCE_GENERIC)) && p.dk == kD &&
           p.dv == kD && scan_tc_supported(p);
}

}  // namespace

int scan_segment_count(const Problem &p, unsigned flags) {
    if (!scan_segmentable(p, flags) || p.B <= 0 || p.T < 2) return 0;
    return dense_segments(p, flags, p.chunk);
}

int scan_varlen_segment_count(const Problem &p, const int *lengths, int n, unsigned flags,
                              std::vector<char> *cut) {
    cut->assign((size_t)std::max(n, 0), 0);
    if (!scan_segmentable(p, flags) || n <= 0) return 0;
    return choose_list_segments(p, lengths, n, flags, p.chunk, cut);
}

size_t scan_segmented_bytes(const Problem &p, int nseq, int P) {
    return plan_scan(p, nseq, P).total;
}

cudaError_t launch_scan_segmented(const Problem &p, const float *records, size_t rec_floats,
                                  const ScanSeq *seqs, int nseq, int P, void *workspace,
                                  cudaStream_t stream) {
    const ScanSegments s = plan_scan(p, nseq, P);
    if (s.P != P || s.total == 0) return cudaErrorInvalidValue;
    const int C = p.chunk;
    for (int i = 0; i < nseq; ++i)
        if (effective_segments(seqs[i].T, P, C) != P) return cudaErrorInvalidValue;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    float *state = reinterpret_cast<float *>(ws + s.off_state);

    std::vector<unsigned char> host(s.table_bytes, 0);
    ScanRun *runA = reinterpret_cast<ScanRun *>(host.data() + s.off_runA);
    ScanRun *runB = reinterpret_cast<ScanRun *>(host.data() + s.off_runB);
    int a = 0, bb = 0;
    for (int b = 0; b < nseq; ++b) {
        const ScanSeq &sq = seqs[b];
        const int base = b * s.group;
        const int per = ((sq.T + C - 1) / C + P - 1) / P;  // chunks per segment
        auto run = [&](int q, int slot_j, int flags) {
            const int c0 = q * per;
            ScanRun r;
            r.tok0 = sq.tok0 + (long long)c0 * C;
            r.rec_base = sq.rec_base + (long long)c0 * sq.c_stride;
            r.T = std::min(sq.T, (q + 1) * per * C) - c0 * C;
            r.slot = base + slot_j;
            r.hv_stride = sq.hv_stride;
            r.c_stride = sq.c_stride;
            r.flags = flags;
            r.pad = 0;
            return r;
        };
        runA[a++] = run(0, 0, p.h0 ? 0 : kRunStartZero);
        for (int q = 1; q <= P - 2; ++q) {
            runA[a++] = run(q, 2 * q - 1, kRunZeroValues | kRunNoOutputs | kRunStartIdentity);  // M_q
            runA[a++] = run(q, 2 * q, kRunNoOutputs | kRunStartZero);                           // c_q
        }
        for (int q = 1; q <= P - 1; ++q) runB[bb++] = run(q, 2 * (q - 1), 0);
    }
    // pageable source: the call returns once the bytes have been taken
    cudaError_t e = cudaMemcpyAsync(ws, host.data(), s.table_bytes, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;

    std::vector<int> sl((size_t)nseq);
    for (int b = 0; b < nseq; ++b) sl[b] = seqs[b].slot;
    if ((e = copy_initial_states(p, state, sl, P, stream)) != cudaSuccess) return e;

    Problem wave = p;
    wave.h0 = state;
    wave.ht = state;
    e = launch_chunk_scan_runs(wave, records, rec_floats,
                               reinterpret_cast<const ScanRun *>(ws + s.off_runA), s.nA, stream);
    if (e != cudaSuccess) return e;
    e = launch_combine(p, state, nseq, P, stream);
    if (e != cudaSuccess) return e;
    e = launch_chunk_scan_runs(wave, records, rec_floats,
                               reinterpret_cast<const ScanRun *>(ws + s.off_runB), s.nB, stream);
    if (e != cudaSuccess) return e;
    return copy_final_states(p, state, sl, P, stream);
}

}  // namespace gdr
