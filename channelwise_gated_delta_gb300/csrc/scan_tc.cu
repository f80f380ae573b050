// scan_tc.cu -- the state scan of the CUDA-core chunked prefill on the tensor
// cores: one CTA per (sequence, value head) carries the dk x dv state from
// chunk to chunk with every contraction a tcgen05 MMA, accumulators and the
// state in tensor memory.
//
// Page "Reorder channelwise gated delta rule chunked hot loops for
// autovectorization" (pytorch/executorch PR #21021), second commit summary:
// the inter-chunk state carry of the chunkwise forward.  Per chunk, from the
// records gdr_chunk_prep leaves (WY pseudo-keys Wk and pseudo-values Wv, the
// decayed queries Qt and keys Kh, the masked P, the decay gam of the chunk),
// with S the state at the chunk start:
//   U = Wv - Wk S,   O = Qt S + P U,   S <- diag(gam) S + Kh^T U.
// Everything is held transposed so that dv (<= 128) runs over the 128
// tensor-memory lanes: Z^T = S^T Wk^T, O^T = S^T Qt^T + U^T P^T,
// X^T = diag-scaled S^T + U^T Kh, with S^T and U^T the A operands read from
// tensor memory and Wk, Qt, P, Kh the B operands in shared memory.
//
// Precision (f32 q/k/v): every operand x is carried as the bf16 pair
// hi = bf16(x), lo = bf16(x - hi) and every product as hi*hi + hi*lo + lo*hi
// (BF16x3; the dropped lo*lo term and the rounding of lo leave about 2^-17
// of |x|), accumulated in f32.  The state itself stays f32 in tensor memory;
// its bf16 pair is rebuilt from it each chunk.  The prep kernel writes Wk,
// Qt, Kh and P straight in this form (gdr_chunk_prep with the TC layout), so
// the scan moves them with bulk copies.
//
// A segmented scan (segments.cu) launches this kernel over a run table
// instead: each run is a stretch of whole chunks with its own first record,
// state slot and flags; a run that gives a segment's map M starts from the
// identity and reads its values as zero (U = -Wk S), and the runs of the
// first wave drop their outputs.
//
// Warps: 0-3 the chain (lane j = value column j: builds the bf16 state pair,
// U = Wv - Z, the final state), 4 the producer (one thread: bulk copies of
// each chunk's operands), 5 the MMA issuer (one thread), 6-9 the writers
// (O^T out of tensor memory and the outputs to global memory, off the
// chain's path).  Kh is double-buffered; Wk and Qt share one buffer
// (stacked, they are one [2C][dk] operand), P and Wv one each.  Per chunk
// the issuer runs [Z^T | S^T Qt^T] = S^T [Wk; Qt]^T (Z and the part of O^T
// that needs only the state pair, one N = 2C product), then, once the chain
// has formed U, the state product and the rest of O^T (U^T P^T, a second
// accumulator); the chain builds the next chunk's state pair as soon as the
// state product is in, and the writers take O^T out.  Every wait is
// bounded: a timeout sets the CTA's abort flag and the library's error
// word, and everyone runs out its loop.
#include <cuda.h>

#include "common.cuh"
#include "sm100_ptx.cuh"

namespace gdr {
namespace {

using namespace sm100;

constexpr int kScWarps = 10;
constexpr int kScThreads = 32 * kScWarps;
constexpr int kScChainThreads = 128;
constexpr int kScProducer = 4;
constexpr int kScIssuer = 5;
constexpr int kScWriter0 = 6;  // warps 6-9: O^T out of tensor memory, the outputs stored
constexpr uint64_t kScWaitNs = 2000000000ull;  // 2 s per wait

// shared memory (bytes from a 1024-byte aligned base); regions sized for
// C <= 64, dk, dv <= 128
constexpr uint32_t kScWq = 0;         // {Wk hi | Qt hi | Wk lo | Qt lo}, each [C][dk] bf16
                                      // K-major: [Wk; Qt] is one [2C][dk] operand
constexpr uint32_t kScKh = 65536;     // [2] x {hi | lo} [C][dk] for Kh (read MN-major)
constexpr uint32_t kScP = 163840;     // hi | lo [C][C]
constexpr uint32_t kScWv = 180224;    // f32 [C][dv]
constexpr uint32_t kScGam = 212992;   // f32 [dk], copied in with Wk and Qt
constexpr uint32_t kScBars = 214016;  // mbarriers
constexpr uint32_t kScSlot = kScBars + 256;
constexpr uint32_t kScAbort = kScSlot + 4;
constexpr uint32_t kScSmem = kScAbort + 4 + 1024;  // + alignment slack
enum {
    SB_WK = 0,   // Wk, Qt and gam copied in (tx)
    SB_KH = 2,   // [2] Kh copied in (tx)
    SB_QP = 4,   // P copied in (tx)
    SB_WV = 5,   // Wv copied in (tx)
    SB_WKF = 6,  // the [Z | O^T] product has read Wk and Qt (commit)
    SB_KHF = 8,  // [2] the state product has read Kh buffer b (commit)
    SB_Z = 10,   // Z^T ready (commit)
    SB_O = 11,   // O^T ready (commit)
    SB_X = 12,   // state product done (commit)
    SB_S = 13,   // chain: bf16 state pair written, state pre-scaled
    SB_U = 14,   // chain: bf16 U pair written
    SB_OF = 15,  // chain: O^T read
    SB_CH = 16,  // chain: Wv and gam read
    SB_COUNT = 17
};
// tensor memory columns
constexpr uint32_t kScTmX = 0;      // f32 state^T [dv lanes][dk]
constexpr uint32_t kScTmShi = 128;  // bf16 pairs of the state^T (A operand)
constexpr uint32_t kScTmSlo = 192;
constexpr uint32_t kScTmZ = 256;    // f32 [Z^T | S^T Qt^T] [dv][2C]: Z, then the first part of O^T
constexpr uint32_t kScTmUhi = 384;  // bf16 pairs of U^T (A operand)
constexpr uint32_t kScTmUlo = 416;
constexpr uint32_t kScTmO2 = 448;   // f32 U^T P^T, the second part of O^T
constexpr uint32_t kScTmCols = 512;

struct ScanTcArgs {
    const float *ws;    // records (TC layout), ChunkLayout floats each
    const float *h0;    // [slots][HV][dk][dv] or null
    void *out;          // [rows][HV][dv], float or bf16
    float *ht;          // [slots][HV][dk][dv] or null
    const int4 *seqs;   // packed batches: {first row, length, slot, first chunk}
    const ScanRun *runs;  // runs of a segmented scan (instead of seqs), or null
    int *err;           // the library's error word
    int T_dense, HV, dk, dv, C, NC_dense;
    size_t rec_floats;
};

__device__ __forceinline__ void sc_pack(float a, float b, uint32_t &hi, uint32_t &lo) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    hi = *reinterpret_cast<uint32_t *>(&h);
    const float2 f = __bfloat1622float2(h);
    __nv_bfloat162 l = __floats2bfloat162_rn(a - f.x, b - f.y);
    lo = *reinterpret_cast<uint32_t *>(&l);
}

template <typename Tout, bool STORE_HT>
__global__ void __launch_bounds__(kScThreads, 1)
    gdr_chunk_scan_tc(const __grid_constant__ ScanTcArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kScBars);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + kScSlot);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kScAbort);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int HV = a.HV, dk = a.dk, dv = a.dv, C = a.C;

    // the sequence: dense batches (b, hv) with records (b, hv, c); packed
    // batches {first row, length, slot, first chunk} with records (chunk, hv)
    const int hv = blockIdx.x % HV, b = blockIdx.x / HV;
    size_t tok0 = (size_t)b * a.T_dense, rec0 = ((size_t)b * HV + hv) * a.NC_dense, rec_step = 1;
    int T = a.T_dense, sl = b, rflags = 0;
    if (a.runs) {
        const ScanRun r = a.runs[b];
        tok0 = (size_t)r.tok0;
        T = r.T;
        sl = r.slot;
        rec0 = (size_t)r.rec_base + (size_t)hv * r.hv_stride;
        rec_step = (size_t)r.c_stride;
        rflags = r.flags;
    } else if (a.seqs) {
        const int4 sd = a.seqs[b];
        tok0 = (size_t)sd.x;
        T = sd.y;
        sl = sd.z;
        rec0 = (size_t)sd.w * HV + hv;
        rec_step = HV;
    }
    const int NC = (T + C - 1) / C;
    const size_t head = (size_t)sl * HV + hv;

    if (tid == 0) {
        for (int i = 0; i < SB_COUNT + 1; ++i)
            mbar_init(&bars[i], (i >= SB_S && i <= SB_CH) ? kScChainThreads : 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tslot, kScTmCols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tslot;
    auto wait = [&](int id, uint32_t parity) {
        if (*abort_flag) return;
        if (!mbar_wait_bounded(&bars[id], parity, kScWaitNs)) {
            *abort_flag = 1;
            if (a.err) atomicExch(a.err, 1);
        }
    };
    const uint32_t tile = (uint32_t)(C * dk * 4);  // a hi | lo operand region, bytes
    const uint32_t half = (uint32_t)(C * dk * 2);  // one bf16 tile of it

    if (warp == kScProducer) {
        // ================= bulk copies of each chunk's operands
        if (lane == 0) {
            int armed[4] = {-1, -1, -1, -1};  // last chunk armed on WK, KH, QP, WV
            for (int c = 0; c < NC && !*abort_flag; ++c) {
                const unsigned char *rec = reinterpret_cast<const unsigned char *>(
                    a.ws + (rec0 + (size_t)c * rec_step) * a.rec_floats);
                const int bf = c & 1;
                if (c >= 1) wait(SB_WKF, (c - 1) & 1);
                if (*abort_flag) break;
                mbar_arrive_expect_tx(&bars[SB_WK], 2 * tile + (uint32_t)(dk * 4));
                bulk_load_1d(smem + kScWq, rec, half, &bars[SB_WK]);                       // Wk hi
                bulk_load_1d(smem + kScWq + 2 * half, rec + half, half, &bars[SB_WK]);     // Wk lo
                bulk_load_1d(smem + kScWq + half, rec + tile, half, &bars[SB_WK]);         // Qt hi
                bulk_load_1d(smem + kScWq + 3 * half, rec + tile + half, half, &bars[SB_WK]);  // Qt lo
                bulk_load_1d(smem + kScGam, rec + 3 * (size_t)tile + (size_t)C * dv * 4 + (size_t)C * C * 4,
                             (uint32_t)(dk * 4), &bars[SB_WK]);
                armed[0] = c;
                if (c >= 2) wait(SB_KHF + bf, ((c - 2) >> 1) & 1);
                if (*abort_flag) break;
                mbar_arrive_expect_tx(&bars[SB_KH + bf], tile);
                bulk_load_1d(smem + kScKh + bf * 32768, rec + 2 * (size_t)tile, tile, &bars[SB_KH + bf]);
                armed[1] = c;
                if (c >= 1) wait(SB_CH, (c - 1) & 1);
                if (*abort_flag) break;
                mbar_arrive_expect_tx(&bars[SB_WV], (uint32_t)(C * dv * 4));
                bulk_load_1d(smem + kScWv, rec + 3 * (size_t)tile, (uint32_t)(C * dv * 4), &bars[SB_WV]);
                armed[3] = c;
                if (c >= 1) wait(SB_O, (c - 1) & 1);
                if (*abort_flag) break;
                mbar_arrive_expect_tx(&bars[SB_QP], (uint32_t)(C * C * 4));
                bulk_load_1d(smem + kScP, rec + 3 * (size_t)tile + (size_t)C * dv * 4,
                             (uint32_t)(C * C * 4), &bars[SB_QP]);
                armed[2] = c;
            }
            if (*abort_flag) {
                // let the copies already armed land before the CTA leaves
                // (bounded: each at most one more wait limit)
                if (armed[0] >= 0) mbar_wait_bounded(&bars[SB_WK], armed[0] & 1, kScWaitNs);
                for (int c2 = armed[1] - 1; c2 <= armed[1]; ++c2)  // both buffers of Kh
                    if (c2 >= 0) mbar_wait_bounded(&bars[SB_KH + (c2 & 1)], (c2 >> 1) & 1, kScWaitNs);
                if (armed[2] >= 0) mbar_wait_bounded(&bars[SB_QP], armed[2] & 1, kScWaitNs);
                if (armed[3] >= 0) mbar_wait_bounded(&bars[SB_WV], armed[3] & 1, kScWaitNs);
            }
        }
    } else if (warp == kScIssuer) {
        // ================= MMA issue (one thread)
        if (lane == 0) {
            const uint32_t idZ = idesc_bf16(128, C, false, false, false);
            const uint32_t idZO = idesc_bf16(128, 2 * C, false, false, false);
            const uint32_t idX = idesc_bf16(128, dk, false, true, false);
            const uint32_t sbase = smem_u32(smem);
            const uint32_t tZ = tmem + kScTmZ, tO2 = tmem + kScTmO2, tX = tmem + kScTmX;
            const uint32_t tSh = tmem + kScTmShi, tSl = tmem + kScTmSlo;
            const uint32_t tUh = tmem + kScTmUhi, tUl = tmem + kScTmUlo;
            bool issued = false;
            for (int c = 0; c < NC && !*abort_flag; ++c) {
                const int bf = c & 1;
                wait(SB_WK, c & 1);
                wait(SB_S, c & 1);
                if (c >= 1) wait(SB_OF, (c - 1) & 1);  // the writers have read O^T of c - 1
                if (*abort_flag) break;
                tc_fence_after_sync();
                // [Z^T | S^T Qt^T] = S^T [Wk; Qt]^T: Z and the part of O^T that
                // needs only the state pair, one N = 2C product
                {
                    const uint32_t w = sbase + kScWq;
                    const uint64_t dh = smem_desc(w, 128, dk * 16), dl = smem_desc(w + 2 * half, 128, dk * 16);
                    for (int ks = 0; ks < dk / 16; ++ks)
                        mma_bf16_ts(tZ, tSh + 8 * ks, dh + (uint64_t)(16 * ks), idZO, ks > 0 ? 1u : 0u);
                    for (int ks = 0; ks < dk / 16; ++ks)
                        mma_bf16_ts(tZ, tSh + 8 * ks, dl + (uint64_t)(16 * ks), idZO, 1u);
                    for (int ks = 0; ks < dk / 16; ++ks)
                        mma_bf16_ts(tZ, tSl + 8 * ks, dh + (uint64_t)(16 * ks), idZO, 1u);
                    mma_commit(&bars[SB_Z]);
                    mma_commit(&bars[SB_WKF]);
                    issued = true;
                }
                // then, with U: X^T += U^T Kh (X pre-scaled by the chain),
                // whose commit also covers the first part of O^T, the last
                // reader of the state pair; then the second part of O^T
                wait(SB_U, c & 1);
                wait(SB_KH + bf, (c >> 1) & 1);
                if (*abort_flag) break;
                tc_fence_after_sync();
                {
                    const uint32_t kh = sbase + kScKh + bf * 32768;
                    const uint64_t hh = smem_desc(kh, dk * 16, 128), hl = smem_desc(kh + half, dk * 16, 128);
                    const uint32_t step = (uint32_t)(32 * dk) >> 4;  // 16 rows of s
                    for (int ks = 0; ks < C / 16; ++ks)
                        mma_bf16_ts(tX, tUh + 8 * ks, hh + (uint64_t)(step * ks), idX, 1u);
                    for (int ks = 0; ks < C / 16; ++ks)
                        mma_bf16_ts(tX, tUh + 8 * ks, hl + (uint64_t)(step * ks), idX, 1u);
                    for (int ks = 0; ks < C / 16; ++ks)
                        mma_bf16_ts(tX, tUl + 8 * ks, hh + (uint64_t)(step * ks), idX, 1u);
                    mma_commit(&bars[SB_X]);
                    mma_commit(&bars[SB_KHF + bf]);
                }
                wait(SB_QP, c & 1);
                if (*abort_flag) break;
                tc_fence_after_sync();
                {
                    const uint32_t p = sbase + kScP;
                    const uint64_t ph = smem_desc(p, 128, C * 16), pl = smem_desc(p + C * C * 2, 128, C * 16);
                    for (int ks = 0; ks < C / 16; ++ks)
                        mma_bf16_ts(tO2, tUh + 8 * ks, ph + (uint64_t)(16 * ks), idZ, ks > 0 ? 1u : 0u);
                    for (int ks = 0; ks < C / 16; ++ks)
                        mma_bf16_ts(tO2, tUh + 8 * ks, pl + (uint64_t)(16 * ks), idZ, 1u);
                    for (int ks = 0; ks < C / 16; ++ks)
                        mma_bf16_ts(tO2, tUl + 8 * ks, ph + (uint64_t)(16 * ks), idZ, 1u);
                    mma_commit(&bars[SB_O]);
                }
            }
            // every MMA issued is done before the tensor memory is released
            if (issued) {
                mma_commit(&bars[SB_COUNT]);
                mbar_wait_bounded(&bars[SB_COUNT], 0, kScWaitNs);
            }
        }
    } else if (warp < 4) {
        // ================= the chain: lane j = value column j
        const int j = tid;
        const bool jv = j < dv;
        const bool vals = jv && !(rflags & kRunZeroValues);    // values read (else zero)
        const uint32_t lo = (uint32_t)(32 * warp) << 16;
        const float *Wv = reinterpret_cast<const float *>(smem + kScWv);
        // the initial state (transposed: lane j holds column j of h0)
        for (int g = 0; g < dk / 16; ++g) {
            uint32_t x[16];
#pragma unroll
            for (int m = 0; m < 16; ++m)
                x[m] = __float_as_uint(
                    (rflags & kRunStartIdentity) ? (16 * g + m == j ? 1.f : 0.f)
                    : (jv && a.h0 && !(rflags & kRunStartZero)) ? a.h0[(head * dk + 16 * g + m) * dv + j]
                                                                : 0.f);
            tmem_st16(tmem + lo + kScTmX + 16 * g, x);
        }
        tmem_st_wait();
        // the state's bf16 pair for chunk cc's products, then the state
        // pre-scaled by that chunk's decay for its update
        auto rebuild = [&](int cc) {
            wait(SB_WK, cc & 1);  // gam of chunk cc
            if (*abort_flag) return;
            tc_fence_after_sync();
            const float *gam = reinterpret_cast<const float *>(smem + kScGam);
            for (int g = 0; g < dk / 16; ++g) {
                float x[16];
                tmem_ld16(tmem + lo + kScTmX + 16 * g, x);
                uint32_t h[8], l[8], xs[16];
#pragma unroll
                for (int m = 0; m < 8; ++m) sc_pack(x[2 * m], x[2 * m + 1], h[m], l[m]);
                tmem_st8(tmem + lo + kScTmShi + 8 * g, h);
                tmem_st8(tmem + lo + kScTmSlo + 8 * g, l);
#pragma unroll
                for (int m = 0; m < 16; ++m) xs[m] = __float_as_uint(x[m] * gam[16 * g + m]);
                tmem_st16(tmem + lo + kScTmX + 16 * g, xs);
            }
            tmem_st_wait();
            tc_fence_before_sync();
            mbar_arrive(&bars[SB_S]);
        };
        if (NC > 0) rebuild(0);
        for (int c = 0; c < NC && !*abort_flag; ++c) {
            const int t0 = c * C, L = min(C, T - t0);
            // U = Wv - Z, as its bf16 pair
            wait(SB_Z, c & 1);
            wait(SB_WV, c & 1);
            if (*abort_flag) break;
            tc_fence_after_sync();
            for (int g = 0; g < C / 16; ++g) {
                float z[16];
                tmem_ld16(tmem + lo + kScTmZ + 16 * g, z);
                uint32_t h[8], l[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const int s = 16 * g + 2 * m;
                    const float u0 = (vals ? Wv[s * dv + j] : 0.f) - z[2 * m];
                    const float u1 = (vals ? Wv[(s + 1) * dv + j] : 0.f) - z[2 * m + 1];
                    sc_pack(u0, u1, h[m], l[m]);
                }
                tmem_st8(tmem + lo + kScTmUhi + 8 * g, h);
                tmem_st8(tmem + lo + kScTmUlo + 8 * g, l);
            }
            tmem_st_wait();
            tc_fence_before_sync();
            mbar_arrive(&bars[SB_U]);
            mbar_arrive(&bars[SB_CH]);
            // the next chunk's state pair as soon as the state product (and
            // with it the first part of O^T) is in
            if (c + 1 < NC) {
                wait(SB_X, c & 1);
                rebuild(c + 1);
            }
        }
        if (STORE_HT && a.ht) {
            if (NC > 0) wait(SB_X, (NC - 1) & 1);
            if (!*abort_flag) {
                tc_fence_after_sync();
                for (int g = 0; g < dk / 16; ++g) {
                    float x[16];
                    tmem_ld16(tmem + lo + kScTmX + 16 * g, x);
#pragma unroll
                    for (int m = 0; m < 16; ++m)
                        if (jv) a.ht[(head * dk + 16 * g + m) * dv + j] = x[m];
                }
            }
        }
    } else if (warp >= kScWriter0) {
        // ================= the writers: warp w reads tensor-memory lanes
        // 32 (w % 4) .., lane j = value column j; each chunk's two parts of
        // O^T summed into registers, their columns freed, then the outputs
        // stored while the chain and the issuer go on
        const int j = 32 * (warp & 3) + lane;
        const bool outs = j < dv && !(rflags & kRunNoOutputs);
        const uint32_t lo = (uint32_t)(32 * (warp & 3)) << 16;
        Tout *out = static_cast<Tout *>(a.out);
        for (int c = 0; c < NC && !*abort_flag; ++c) {
            const int t0 = c * C, L = min(C, T - t0);
            wait(SB_O, c & 1);
            if (*abort_flag) break;
            tc_fence_after_sync();
            float o[64];
#pragma unroll
            for (int g = 0; g < 4; ++g)
                if (16 * g < C) {
                    float og[16], og2[16];
                    tmem_ld16(tmem + lo + kScTmZ + C + 16 * g, og);
                    tmem_ld16(tmem + lo + kScTmO2 + 16 * g, og2);
#pragma unroll
                    for (int m = 0; m < 16; ++m) o[16 * g + m] = og[m] + og2[m];
                }
            tc_fence_before_sync();
            mbar_arrive(&bars[SB_OF]);
            if (outs) {
#pragma unroll
                for (int s = 0; s < 64; ++s)
                    if (s < L) out[((tok0 + t0 + s) * HV + hv) * dv + j] = from_f32<Tout>(o[s]);
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, kScTmCols);
}

}  // namespace

// f32 (or bf16) outputs; records in the TC layout (gdr_chunk_prep<..., TCREC>).
bool scan_tc_supported(const Problem &p) {
    return (p.dk == 32 || p.dk == 64 || p.dk == 128) && (p.dv == 32 || p.dv == 64 || p.dv == 128) &&
           (p.chunk == 16 || p.chunk == 32 || p.chunk == 64);
}

namespace {
cudaError_t launch_scan(const Problem &p, const float *records, size_t rec_floats,
                        const int4 *seqs, const ScanRun *runs, long long units,
                        cudaStream_t stream) {
    int *err = nullptr;
    cudaError_t e = device_error_word(&err);
    if (e != cudaSuccess) return e;
    ScanTcArgs a;
    a.ws = records; a.h0 = p.h0; a.out = p.out; a.ht = p.ht; a.seqs = seqs; a.runs = runs;
    a.err = err;
    a.T_dense = p.T; a.HV = p.HV; a.dk = p.dk; a.dv = p.dv; a.C = p.chunk;
    a.NC_dense = (p.T + p.chunk - 1) / p.chunk;
    a.rec_floats = rec_floats;
    const long long ctas = units * p.HV;
    if (ctas == 0) return cudaSuccess;
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    trace_begin(kKernChunkScanTc, stream);
    if (p.bf16) {
        auto k = p.ht ? gdr_chunk_scan_tc<__nv_bfloat16, true> : gdr_chunk_scan_tc<__nv_bfloat16, false>;
        if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kScSmem)) != cudaSuccess)
            return e;
        k<<<(unsigned)ctas, kScThreads, kScSmem, stream>>>(a);
    } else {
        auto k = p.ht ? gdr_chunk_scan_tc<float, true> : gdr_chunk_scan_tc<float, false>;
        if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kScSmem)) != cudaSuccess)
            return e;
        k<<<(unsigned)ctas, kScThreads, kScSmem, stream>>>(a);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    trace_end(kKernChunkScanTc, stream);
    return cudaSuccess;
}
}  // namespace

cudaError_t launch_chunk_scan_tc(const Problem &p, const float *records, size_t rec_floats,
                                 const int4 *seqs, int nseq, cudaStream_t stream) {
    return launch_scan(p, records, rec_floats, seqs, nullptr, seqs ? nseq : p.B, stream);
}

cudaError_t launch_chunk_scan_runs(const Problem &p, const float *records, size_t rec_floats,
                                   const ScanRun *runs, int nrun, cudaStream_t stream) {
    return launch_scan(p, records, rec_floats, nullptr, runs, nrun, stream);
}

}  // namespace gdr
