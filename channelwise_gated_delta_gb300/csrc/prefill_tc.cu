// prefill_tc.cu -- chunkwise WY/UT prefill on the Blackwell tensor cores
// (tcgen05 MMA, TMEM accumulators, TMA) for bf16 q/k/v with dk = dv = 128 and
// chunks of 64 tokens: one warp-specialised CTA per (sequence, value head),
// the float32 state resident in tensor memory.
//
// Method: page "Reorder channelwise gated delta rule chunked hot loops for
// autovectorization" (pytorch/executorch PR #21021), second commit summary --
// per chunk: per-channel log-decay prefix sums, the causal query/key terms,
// the beta-folded unit-lower triangular transform, WY pseudo-values, and the
// state carried to the next chunk, with a ragged last chunk through the same
// code.  The triangular transform is a block forward substitution (16 x 16
// diagonal-block inverses, then the off-diagonal blocks by small matrix
// products), the block-TRSM structure of trymirai/uzu PR #576 ("Support
// TreeUpdateSolve kernel", commit summary).
//
// Algebra per chunk of L <= 64 tokens (r, s local token indices; S the state
// at the chunk start; G the inclusive per-channel prefix sum of g):
//   A[r,s] = beta_r sum_i k_ri k_si exp(G_ri - G_si)   (s < r)
//   P[r,s] =        sum_i q_ri k_si exp(G_ri - G_si)   (s <= r)
//   T'     = (I + A)^-1 diag(beta)
//   U      = T' (V - (exp(G) * K) S)
//   O      = (exp(G) * Q) S + P U
//   S     <- diag(exp(G_L)) S + (exp(G_L - G) * K)^T U
// Factoring around a reference row m of the chunk, with
//   Lk = K * exp(G - G_m),  Lq = Q * exp(G - G_m),  R = K * exp(G_m - G),
//   S' = diag(exp(G_m)) S:
//   A = tril(diag(beta) Lk R^T),  P = tril(Lq R^T),  Z = Lk S',
//   U = T' (V - Z),  O = Lq S' + P U,
//   S'_next = diag(c) (S' + R^T U),  c = exp(G'_m + G_L - G_m)
// (G'_m the next chunk's reference row; G is kept in log2 units so that every
// factor is one ex2).  The same factor c multiplies both terms, so the state
// update is an accumulation X += U^T R on the tensor core followed by one
// column scaling, where X = S'^T is the state kept in TMEM.
// While no 16-row quarter of the chunk decays by more than 80/3 nats and no
// half by more than 43 nats in any channel, every factor lies within
// exp(+-80) and c above exp(-86), in the normal float range.  A chunk outside
// that range uses m := the chunk start (Lk = exp(G) K, Lq = exp(G) Q,
// R = exp(G_L - G) K, all factors <= 1) with A and P built 16 x 16 block by
// block on bf16 mma.sync, each block's decays split about a row inside it
// (exact_block below; pairwise decays for a diagonal block past that
// range); its carry is X <- (exp(G_L) X + U^T R) c, the first factor applied
// when X is written, so the result is right for any g <= 0.
//
// GB300 mapping: one CTA of 20 warps per (sequence, value head) walks that
// head's chunks in order.
//   warps 0-7   chain warps: read back -Z, U and the state from TMEM between
//               the state-dependent MMAs, scale the state by c, write the bf16
//               operands S'^T, -Z^T and U^T back into TMEM, and store O.
//   warps 8-15  prep warps: the prefix sums, range check and carry factors,
//               the bf16 operand tiles Lq, Lk, R of the next chunk, the P
//               read-back, and the exact path's A and P blocks.
//   warp 16     producer: TMA loads of k, q, g and v, and the gram
//               [Lq; Lk] R^T of the chunk being prepared.
//   warp 17     issues the state-dependent MMAs of the chunk being scanned:
//               Z^T = S'^T Lk^T, O^T = S'^T Lq^T, U^T = (V^T - Z^T) T'^T,
//               then X^T += U^T R and O^T += U^T P^T.
//   warps 18-19 invert I + A for the chunk being prepared (its A rows are
//               TMEM lanes 64-127, the lane quarters of these two warps).
// Preparation of chunk c+1 starts with its prefix sums and carry factors as
// soon as its k, q, g tiles land, and writes its operand tiles once chunk c's
// O^T product has read theirs, so the prefix sums, tiles, gram and inverse of
// the next chunk overlap the state chain of the current one.  Every state
// product is transposed so that M = dv = 128 fills the MMA; the state-side A
// operands are bf16 in TMEM.  Every mbarrier wait is bounded.
#include <cuda.h>
#include <string.h>

#include "common.cuh"
#include "sm100_ptx.cuh"
#include "tma_host.h"

namespace gdr {
namespace {

using namespace sm100;

constexpr int kC = 64;      // chunk length
constexpr int kD = 128;     // dk = dv
constexpr int kWarps = 20;            // 5 per SM sub-partition: 96 registers a thread
constexpr int kThreads = 32 * kWarps;
constexpr int kWarpPrep0 = 8;        // warps 8-15
constexpr int kWarpProducer = 16;    // TMA loads and the gram MMA
constexpr int kWarpChainIssuer = 17;
constexpr int kWarpSolver0 = 18;     // warps 18-19
constexpr int kChainThreads = 256;
constexpr int kPrepThreads = 256;
constexpr int kHandThreads = kChainThreads + 32;  // chain warps + chain issuer warp
// named barriers
constexpr int kNbS = 1;      // chain -> issuer: X and S'^T of the next chunk written
constexpr int kNbZb = 2;     // chain -> issuer: -Z^T written
constexpr int kNbUb = 3;     // chain -> issuer: U^T written
constexpr int kNbOfree = 4;  // chain -> issuer: O^T read
constexpr int kNbPrep = 5;   // prep warps
constexpr int kNbSolve = 6;  // solver warps

constexpr float kLog2e = 1.4426950408889634f;
// Fast-path decay limits (log2 units): a 16-row quarter within a third of 80
// nats keeps the operand factors within exp(+-80); a half chunk within 43
// nats keeps the carry factor c, which spans the second half of one chunk and
// the first half of the next, above exp(-86).
constexpr float kQuarterLog2 = 80.f / 3.f * kLog2e;
constexpr float kHalfLog2 = 43.f * kLog2e;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait

// ---- shared memory map (bytes from a 1024-byte aligned base)
constexpr uint32_t kRawK = 0;              // k: 2 TMA boxes [64 rows][64 bf16], 128B-swizzled
constexpr uint32_t kRawQ = 16384;          // q: same
constexpr uint32_t kG = 32768;             // g: 4 boxes [64 rows][32 f32], 128B-swizzled; then G
constexpr uint32_t kOpV = 65536;           // v: 2 boxes [64 s][64 j] = swizzled MN-major A operand
constexpr uint32_t kOpL = 81920;           // [128][128] K-major: rows 0-63 Lq, 64-127 Lk
constexpr uint32_t kOpR = 114688;          // [2][64][128] K-major: R (by chunk parity)
constexpr uint32_t kOpP = 147456;          // P as K-major B [64 r][64 s]
constexpr uint32_t kOpT = 155648;          // T' as K-major B [64 r][64 s]
constexpr uint32_t kA32 = 163840;          // f32 A (64 x 64, swizzled)
constexpr uint32_t kT32 = 180224;          // f32 T
constexpr uint32_t kX32 = 196608;          // f32 [4][16][16] solve scratch
constexpr uint32_t kStage = 200704;        // bf16 O staging: per chain warp one [32 r][32 j] box
constexpr uint32_t kTot = 217088;          // f32 [8][128] per-warp prefix totals
constexpr uint32_t kGm = 221184;           // f32 [2][128] G at the reference row (by chunk parity)
constexpr uint32_t kGL = kGm + 1024;       // f32 [2][128] G at the last row
constexpr uint32_t kCv = kGL + 1024;       // f32 [2][128] carry factor c of the chunk scanned
constexpr uint32_t kAv = kCv + 1024;       // f32 [2][128] pre-scale of the next chunk's X
constexpr uint32_t kGsc = kAv + 1024;      // f32 [64] scalar gate: G of the chunk prepared
constexpr uint32_t kBeta = kGsc + 256;     // f32 [64] beta of the chunk being inverted
constexpr uint32_t kBars = kBeta + 256;    // mbarriers
enum {
    MB_RAW = 0,  // k, q, g tiles landed (TMA)
    MB_V,        // v tile landed (TMA)
    MB_TILES,    // operand tiles, carry factors, slow flag of a chunk written (prep)
    MB_GRAM,     // gram complete, or the exact path's A and P written
    MB_GFREE,    // gram read back and A consumed (solvers, P readers)
    MB_TP,       // T' and P written (solvers, P readers)
    MB_Z,        // Z^T product complete
    MB_OPART,    // O^T = S'^T Lq^T complete: the Lq, Lk tiles are free
    MB_U,        // U^T product complete: T' and v buffers free
    MB_X,        // state and output accumulations complete
    kNumBars
};
constexpr uint32_t kTmemSlot = kBars + 8 * kNumBars;
constexpr uint32_t kAbort = kTmemSlot + 4;   // i32 sticky abort flag
constexpr uint32_t kSlowFlag = kAbort + 4;   // i32 [2] (by chunk parity)
constexpr uint32_t kSmemUsed = kSlowFlag + 8;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // + alignment slack for the 1024-byte base
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kTot >= kStage + 16384, "layout");
constexpr uint32_t kBytesKQG = 16384 + 16384 + 32768;
constexpr uint32_t kBytesV = 16384;

// ---- TMEM columns (float32 accumulators, lane = M row)
constexpr uint32_t kTmGram = 0;   // [128 x 64]: rows 0-63 Lq R^T (P), 64-127 Lk R^T (A)
constexpr uint32_t kTmZ = 64;     // [128 j x 64 r]  Z^T
constexpr uint32_t kTmU = 128;    // [128 j x 64 r]  U^T
constexpr uint32_t kTmO = 192;    // [128 j x 64 r]  O^T
constexpr uint32_t kTmX = 256;    // [128 j x 128 i] the state X = S'^T
constexpr uint32_t kTmSb = 384;   // S'^T as bf16 A operand, 2 per column
constexpr uint32_t kTmUb = 448;   // U^T as bf16 A operand
constexpr uint32_t kTmZb = 480;   // -Z^T as bf16 A operand
constexpr uint32_t kTmemCols = 512;

// 64 x 64 f32 tiles (A, T) with an XOR swizzle: rows and columns both walk
// conflict-free
__device__ __forceinline__ int sq_idx(int r, int s) { return r * 64 + (s ^ (r & 31)); }
// The diagonal blocks of A are only read by the diagonal inverses, so they
// are stored transposed: A[16 I + p][16 I + q] at row 16 I + q, slot p, and
// column q of a block is one contiguous run of 16 floats.
__device__ __forceinline__ int diagT_idx(int I, int q, int p) { return (16 * I + q) * 64 + 32 * (I >> 1) + p; }
// byte offset of bf16 element (r, i) of a k or q tile (two 64-channel boxes)
__device__ __forceinline__ uint32_t kq_off(int r, int i) {
    return (uint32_t)((i >> 6) * 8192 + r * 128 + ((((i & 63) >> 3) ^ (r & 7)) << 4) + (i & 7) * 2);
}
// byte offset of f32 element (r, i) of the g tile (four 32-channel boxes)
__device__ __forceinline__ uint32_t g_off(int r, int i) {
    return (uint32_t)((i >> 5) * 8192 + r * 128 + ((((i & 31) >> 2) ^ (r & 7)) << 4) + (i & 3) * 4);
}

__device__ __forceinline__ uint4 pack_bf16x8(const float *x) {
    uint4 u;
    __nv_bfloat162 h0 = __floats2bfloat162_rn(x[0], x[1]);
    __nv_bfloat162 h1 = __floats2bfloat162_rn(x[2], x[3]);
    __nv_bfloat162 h2 = __floats2bfloat162_rn(x[4], x[5]);
    __nv_bfloat162 h3 = __floats2bfloat162_rn(x[6], x[7]);
    u.x = *reinterpret_cast<uint32_t *>(&h0);
    u.y = *reinterpret_cast<uint32_t *>(&h1);
    u.z = *reinterpret_cast<uint32_t *>(&h2);
    u.w = *reinterpret_cast<uint32_t *>(&h3);
    return u;
}
__device__ __forceinline__ void unpack_bf16x8(uint4 u, float *x) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162 *>(&w[e]);
        float2 f = __bfloat1622float2(h);
        x[2 * e] = f.x;
        x[2 * e + 1] = f.y;
    }
}
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ float2 unpack_bf16x2(uint32_t w) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w));
}

// D (+)= A * B^T with shared-memory operands, K_STEPS steps of K = 16; each
// step advances the descriptors' start-address field (address / 16) by a
// fixed number of bytes, which never carries out of the field inside shared
// memory.
template <int K_STEPS>
__device__ __forceinline__ void gemm_ss(uint32_t d_tmem, uint64_t a_desc, uint32_t a_step,
                                        uint64_t b_desc, uint32_t b_step, uint32_t idesc,
                                        bool accumulate_first) {
#pragma unroll
    for (int ks = 0; ks < K_STEPS; ++ks)
        mma_bf16(d_tmem, a_desc + (uint64_t)((ks * a_step) >> 4),
                 b_desc + (uint64_t)((ks * b_step) >> 4), idesc,
                 (ks > 0 || accumulate_first) ? 1u : 0u);
}
// Same with the A operand in tensor memory (bf16 packed two per column,
// eight columns per K-step of 16).
template <int K_STEPS>
__device__ __forceinline__ void gemm_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                        uint32_t b_step, uint32_t idesc, bool accumulate_first) {
#pragma unroll
    for (int ks = 0; ks < K_STEPS; ++ks)
        mma_bf16_ts(d_tmem, a_tmem + 8 * ks, b_desc + (uint64_t)((ks * b_step) >> 4), idesc,
                    (ks > 0 || accumulate_first) ? 1u : 0u);
}

// Bounded wait on an mbarrier phase.  A timeout sets the CTA's sticky abort
// flag; later waits then return at once, nothing new is issued, and every
// group runs out its loop, so a stuck copy or MMA can never hang the kernel.
__device__ __forceinline__ void wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
    if (*abort_flag) return;
    if (!mbar_wait_bounded(bar, parity, kWaitLimitNs)) *abort_flag = 1;
}

// ---- tf32 mma.sync for the 16 x 16 block products of the inverse
__device__ __forceinline__ void mma_tf32(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Block (I, J) of a swizzled 64 x 64 f32 tile: with R = 16 I + r, element
// (r, c) sits at R * 64 + 16 (J ^ (I & 1)) + (c ^ r).
__device__ __forceinline__ const float *swz_block(const float *tile, int I, int J) {
    return tile + I * 1024 + 16 * (J ^ (I & 1));
}
struct FragOffsets {  // per-lane offsets of the m16n8k8 tf32 fragments in a swizzled block
    int a0, a1;       // A: row gq, columns tq / tq + 4
    int b0, b1;       // B: rows tq / tq + 4, column gq
    int x0, x1;       // the same for a plain [16][16] block (row stride 16)
};
__device__ __forceinline__ FragOffsets frag_offsets(int lane) {
    const int gq = lane >> 2, tq = lane & 3;
    FragOffsets f;
    f.a0 = gq * 64 + (tq ^ gq);
    f.a1 = gq * 64 + ((tq + 4) ^ gq);
    f.b0 = tq * 64 + (tq ^ gq);
    f.b1 = (tq + 4) * 64 + ((tq + 4) ^ gq);
    f.x0 = tq * 16 + gq;
    f.x1 = (tq + 4) * 16 + gq;
    return f;
}
// acc += X * Y for 16 x 16 blocks on tf32 mma.sync (one warp); X a swizzled
// block, Y a swizzled block (SWZ_Y) or a plain [16][16] scratch block.
template <bool SWZ_Y>
__device__ __forceinline__ void blk_mma2(float (&acc)[2][4], const float *X, const float *Y,
                                         const FragOffsets &f) {
#pragma unroll
    for (int kh = 0; kh < 2; ++kh) {
        uint32_t a[4];
        a[0] = __float_as_uint(X[f.a0 + 8 * kh]);
        a[1] = __float_as_uint(X[f.a0 + 512 + 8 * (kh ^ 1)]);
        a[2] = __float_as_uint(X[f.a1 + 8 * kh]);
        a[3] = __float_as_uint(X[f.a1 + 512 + 8 * (kh ^ 1)]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            uint32_t b0, b1;
            if (SWZ_Y) {
                b0 = __float_as_uint(Y[f.b0 + 512 * kh + 8 * (nt ^ kh)]);
                b1 = __float_as_uint(Y[f.b1 + 512 * kh + 8 * (nt ^ kh)]);
            } else {
                b0 = __float_as_uint(Y[f.x0 + 128 * kh + 8 * nt]);
                b1 = __float_as_uint(Y[f.x1 + 128 * kh + 8 * nt]);
            }
            mma_tf32(acc[nt], a, b0, b1);
        }
    }
}
__device__ __forceinline__ void blk_store(float *xs, const float (&acc)[2][4], int lane) {
    const int gq = lane >> 2, tq = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        xs[gq * 16 + 8 * nt + 2 * tq] = acc[nt][0];
        xs[gq * 16 + 8 * nt + 2 * tq + 1] = acc[nt][1];
        xs[(gq + 8) * 16 + 8 * nt + 2 * tq] = acc[nt][2];
        xs[(gq + 8) * 16 + 8 * nt + 2 * tq + 1] = acc[nt][3];
    }
}

// ---- exact path: the intra-chunk matrices A and P block by block
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Diagonal blocks about their middle row: every factor within exp(+-60)
// (log2 units).
constexpr float kDiagLog2 = 60.f * kLog2e;

// One warp: rows r0 .. r0 + 15 of A and P against nt_n 8-column tiles from
// column s0, on bf16 m16n8k16 mma.sync over the 128 key channels.  The
// decay of a pair splits at reference row b,
//   exp(G_r - G_s) = exp(G_r - G_b) exp(G_b - G_s),
// the first factor scaling the row operands k_r and q_r and the second the
// column operand k_s (both <= 1 when s < b <= r).  SCALAR_G: one decay per
// row, applied to each product instead.  Writes every element of its blocks
// (zeros above the diagonal and past row L); skip: zeros only.
template <bool SCALAR_G>
__device__ __forceinline__ void exact_block(const unsigned char *smem, float *sA, unsigned char *opP,
                                            int r0, int s0, int nt_n, int b, bool diag, bool skip,
                                            int L, float br0, float br1, int lane) {
    const int gq = lane >> 2, tq = lane & 3;
    float acc_a[4][4], acc_p[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc_a[nt][e] = acc_p[nt][e] = 0.f;
    if (!skip) {
#pragma unroll 1
        for (int ks = 0; ks < 8; ++ks) {
            const int chs[2] = {16 * ks + 2 * tq, 16 * ks + 2 * tq + 8};
            float2 gb[2];
            if (!SCALAR_G) {
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    gb[h] = *reinterpret_cast<const float2 *>(smem + kG + g_off(b, chs[h]));
            }
            // row operands: register (2 h + i) holds row r0 + gq + 8 i, channels chs[h]
            uint32_t ak[4], aq[4];
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int r = r0 + gq + 8 * i;
                    const uint32_t kw = *reinterpret_cast<const uint32_t *>(smem + kRawK + kq_off(r, chs[h]));
                    const uint32_t qw = *reinterpret_cast<const uint32_t *>(smem + kRawQ + kq_off(r, chs[h]));
                    if (SCALAR_G) {
                        ak[2 * h + i] = kw;
                        aq[2 * h + i] = qw;
                    } else {
                        const float2 g = *reinterpret_cast<const float2 *>(smem + kG + g_off(r, chs[h]));
                        const float ex = fast_exp2(g.x - gb[h].x), ey = fast_exp2(g.y - gb[h].y);
                        const float2 kf = unpack_bf16x2(kw), qf = unpack_bf16x2(qw);
                        ak[2 * h + i] = pack_bf16x2(kf.x * ex, kf.y * ey);
                        aq[2 * h + i] = pack_bf16x2(qf.x * ex, qf.y * ey);
                    }
                }
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                if (nt < nt_n) {
                    const int s = s0 + 8 * nt + gq;
                    uint32_t bw[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t kw = *reinterpret_cast<const uint32_t *>(smem + kRawK + kq_off(s, chs[h]));
                        if (SCALAR_G) {
                            bw[h] = kw;
                        } else {
                            const float2 g = *reinterpret_cast<const float2 *>(smem + kG + g_off(s, chs[h]));
                            const float2 kf = unpack_bf16x2(kw);
                            bw[h] = pack_bf16x2(kf.x * fast_exp2(gb[h].x - g.x), kf.y * fast_exp2(gb[h].y - g.y));
                        }
                    }
                    mma_bf16_16816(acc_a[nt], ak, bw[0], bw[1]);
                    mma_bf16_16816(acc_p[nt], aq, bw[0], bw[1]);
                }
            }
        }
    }
    const float *gsv = reinterpret_cast<const float *>(smem + kGsc);
    const int I = r0 >> 4;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
        if (nt >= nt_n) break;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int r = r0 + gq + 8 * i, s = s0 + 8 * nt + 2 * tq;
            const float br = i ? br1 : br0;
            float va[2], vp[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float a = acc_a[nt][2 * i + e], p = acc_p[nt][2 * i + e];
                if (SCALAR_G && !skip) {
                    const float f = fast_exp2(gsv[r] - gsv[s + e]);
                    a *= f;
                    p *= f;
                }
                const bool in = r < L && s + e <= r;
                va[e] = (in && s + e < r) ? br * a : 0.f;
                vp[e] = in ? p : 0.f;
            }
            if (diag) {
                sA[diagT_idx(I, (s & 15), r & 15)] = va[0];
                sA[diagT_idx(I, (s & 15) + 1, r & 15)] = va[1];
            } else {
                sA[sq_idx(r, s)] = va[0];
                sA[sq_idx(r, s + 1)] = va[1];
            }
            *reinterpret_cast<uint32_t *>(opP + kmajor_off(r, s, kC)) = pack_bf16x2(vp[0], vp[1]);
        }
    }
}

struct TileMaps {
    CUtensorMap k, q, g, v, o;
};

// Packed variable-length batches (VARLEN): one record per sequence, {first
// token row in the packed tensors, length, state slot}; the sequence's tensor
// maps sit at the same index of a TileMaps array in global memory.
// SCALAR_G: g is one log-decay per token and value head (gsc, [rows][HV]),
// the same for every key channel.
template <bool HAS_H0, bool STORE_HT, bool VARLEN, bool SCALAR_G>
__global__ void __launch_bounds__(kThreads, 1)
    gdr_prefill_tc_kernel(const __grid_constant__ TileMaps tm, const TileMaps *seq_maps,
                          const int4 *seqs, const float *__restrict__ beta,
                          const float *__restrict__ gsc, const float *h0, float *ht, int T_dense,
                          int HK, int HV, int *dev_error) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int head = blockIdx.x;    // b * HV + hv (b: the sequence's index)
    const int hv = head % HV;
    int b = head / HV;              // batch coordinate of the tensor maps
    const int hk = hv / (HV / HK);
    int T = T_dense;
    size_t tok0 = (size_t)b * T;    // the sequence's first token row
    size_t shead = head;            // state slot * HV + hv
    int start = 0;                  // kSeqStartZero / kSeqStartIdentity, else h0
    const TileMaps *mp = &tm;
    if (VARLEN) {
        const int4 sd = seqs[b];
        tok0 = (size_t)sd.x;
        T = sd.y;
        shead = (size_t)sd.z * HV + hv;
        start = sd.w;
        mp = seq_maps + b;
        b = 0;  // each sequence's maps describe a [1][T][H][128] tensor
    }
    const TileMaps &m = *mp;
    const int NC = (T + kC - 1) / kC;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kBars);
    auto bar = [&](int i) { return bars + i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kTmemSlot);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kAbort);
    volatile int *slow_flag = reinterpret_cast<volatile int *>(smem + kSlowFlag);
    auto vec = [&](uint32_t base, int slot) { return reinterpret_cast<float *>(smem + base) + 128 * slot; };
    auto wait = [&](int i, int chunk) { wait_bar(bar(i), (uint32_t)(chunk & 1), abort_flag); };

    if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
    if (tid == 0) {
        mbar_init(bar(MB_RAW), 1);
        mbar_init(bar(MB_V), 1);
        mbar_init(bar(MB_TILES), 1);
        mbar_init(bar(MB_GRAM), 1);
        mbar_init(bar(MB_GFREE), 1 + 4);  // one solver thread + the four P-reading warps
        mbar_init(bar(MB_TP), 1 + 4);
        mbar_init(bar(MB_Z), 1);
        mbar_init(bar(MB_OPART), 1);
        mbar_init(bar(MB_U), 1);
        mbar_init(bar(MB_X), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    // T' is lower triangular: its strictly-upper 16 x 16 blocks stay zero
    for (int idx = tid; idx < 64 * 8; idx += kThreads) {
        const int r = idx >> 3, s0 = (idx & 7) * 8;
        if ((s0 >> 4) > (r >> 4))
            *reinterpret_cast<uint4 *>(smem + kOpT + kmajor_off(r, s0, kC)) = make_uint4(0, 0, 0, 0);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);  // this warp's lane quarter
    const uint32_t io = idesc_bf16(128, 64, false, false, false);
    int issued_raw = 0, issued_v = 0;  // producer: copies issued on MB_RAW, MB_V

    if (warp < kWarpPrep0) {
        // ================= chain warps: lane quarter wq, half hh of the state
        // columns (i in [64 hh, 64 hh + 64)) and of the chunk rows (r in
        // [32 hh, 32 hh + 32))
        const int wq = warp & 3, hh = warp >> 2;
        const int j = 32 * wq + lane;  // this thread's value column (TMEM lane)
        if (VARLEN && lane == 0) fence_tensormap_acquire(&m.o);
        __nv_bfloat16 *stg = reinterpret_cast<__nv_bfloat16 *>(smem + kStage + 2048 * warp);
        auto handoff = [&](int id) {
            tc_fence_before_sync();
            if (*abort_flag)
                named_sync(id, kHandThreads);
            else
                named_arrive(id, kHandThreads);
        };
        // Writes the state columns i0 .. i0 + 31 from x (the accumulated
        // X + U^T R, or h0): S' = x c is the bf16 operand of the next chunk and
        // X = S' a the stored state; after the last chunk S' is the final state.
        auto put_state = [&](int i0, float (&x)[32], int slot, bool last) {
            const float *cv = vec(kCv, slot) + i0;
            const float *av = vec(kAv, slot) + i0;
            uint32_t wb[16];
#pragma unroll
            for (int u = 0; u < 32; u += 4) {
                const float4 c4 = *reinterpret_cast<const float4 *>(cv + u);
                const float4 a4 = *reinterpret_cast<const float4 *>(av + u);
                const float2 y0 = __fmul2_rn(make_float2(x[u], x[u + 1]), make_float2(c4.x, c4.y));
                const float2 y1 = __fmul2_rn(make_float2(x[u + 2], x[u + 3]), make_float2(c4.z, c4.w));
                wb[u / 2] = pack_bf16x2(y0.x, y0.y);
                wb[u / 2 + 1] = pack_bf16x2(y1.x, y1.y);
                const float2 z0 = __fmul2_rn(y0, make_float2(a4.x, a4.y));
                const float2 z1 = __fmul2_rn(y1, make_float2(a4.z, a4.w));
                x[u] = z0.x;
                x[u + 1] = z0.y;
                x[u + 2] = z1.x;
                x[u + 3] = z1.y;
            }
            if (last) {  // the final factor's a is 1: x holds the final state
                if (STORE_HT && !*abort_flag) {
#pragma unroll
                    for (int u = 0; u < 32; ++u) ht[(shead * kD + i0 + u) * kD + j] = x[u];
                }
            } else {
                uint32_t wx[32];
#pragma unroll
                for (int u = 0; u < 32; ++u) wx[u] = __float_as_uint(x[u]);
                tmem_st32(tl + kTmX + i0, wx);
                tmem_st16(tl + kTmSb + i0 / 2, wb);
            }
        };
        // initial state: X = h0 c a with the factors of the first chunk
        wait(MB_TILES, 0);
#pragma unroll 1
        for (int p = 0; p < 2; ++p) {
            const int i0 = 64 * hh + 32 * p;
            float x[32];
#pragma unroll
            for (int u = 0; u < 32; ++u)
                x[u] = (start & kSeqStartIdentity) ? (i0 + u == j ? 1.f : 0.f)
                       : (HAS_H0 && !(start & kSeqStartZero)) ? h0[(shead * kD + i0 + u) * kD + j]
                                                               : 0.f;
            put_state(i0, x, 1, false);
        }
        tmem_st_wait();
        handoff(kNbS);
#pragma unroll 1
        for (int c = 0; c < NC; ++c) {
            const bool last = c + 1 == NC;
            // -Z^T as the bf16 A operand of the U product
            wait(MB_Z, c);
            tc_fence_after_sync();
            {
                float d[32];
                tmem_ld32(tl + kTmZ + 32 * hh, d);
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) w[e] = pack_bf16x2(-d[2 * e], -d[2 * e + 1]);
                tmem_st16(tl + kTmZb + 16 * hh, w);
                tmem_st_wait();
            }
            handoff(kNbZb);
            // U^T as the bf16 A operand of the state and output products
            wait(MB_U, c);
            tc_fence_after_sync();
            {
                float d[32];
                tmem_ld32(tl + kTmU + 32 * hh, d);
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) w[e] = pack_bf16x2(d[2 * e], d[2 * e + 1]);
                tmem_st16(tl + kTmUb + 16 * hh, w);
                tmem_st_wait();
            }
            handoff(kNbUb);
            // the state: X + U^T R scaled into the next chunk's frame
            wait(MB_X, c);
            tc_fence_after_sync();
            if (!last) wait(MB_TILES, c + 1);  // the carry factors come with the next chunk's tiles
#pragma unroll 1
            for (int p = 0; p < 2; ++p) {
                const int i0 = 64 * hh + 32 * p;
                float x[32];
                tmem_ld32(tl + kTmX + i0, x);
                put_state(i0, x, c & 1, last);
            }
            if (!last) {
                tmem_st_wait();
                handoff(kNbS);
            }
            // O^T -> this warp's bf16 box [32 r][32 j] -> one TMA store
            {
                float o[32];
                tmem_ld32(tl + kTmO + 32 * hh, o);
                if (!last) handoff(kNbOfree);
                if (lane == 0) bulk_wait_read_all();  // the previous store has read the box
                __syncwarp();
#pragma unroll
                for (int u = 0; u < 32; u += 2) {
                    const __nv_bfloat162 h = __floats2bfloat162_rn(o[u], o[u + 1]);
                    stg[u * 32 + lane] = h.x;
                    stg[(u + 1) * 32 + lane] = h.y;
                }
                fence_async_smem();
                __syncwarp();
                // rows past the end of the sequence fall outside the tensor and are dropped
                if (lane == 0 && !*abort_flag) {
                    tma_store_4d(&m.o, stg, 32 * wq, hv, c * kC + 32 * hh, b);
                    bulk_commit_group();
                }
            }
        }
        if (lane == 0) bulk_wait_all();
    } else if (warp < kWarpProducer) {
        // ================= prep warps
        const int pw = warp - kWarpPrep0;  // 0..7
        const int pt = tid - 32 * kWarpPrep0;
        const bool p_reader = (warp & 3) < 2;  // TMEM lanes 0-63: the P rows of the gram
        float gs0 = 0.f, gs1 = 0.f;            // scalar gate: this lane's two log-decays of the chunk
        auto load_gsc = [&](int t0) {
            if (SCALAR_G && pw == 0) {
                gs0 = t0 + 2 * lane < T ? gsc[(tok0 + t0 + 2 * lane) * HV + hv] : 0.f;
                gs1 = t0 + 2 * lane + 1 < T ? gsc[(tok0 + t0 + 2 * lane + 1) * HV + hv] : 0.f;
            }
        };
        load_gsc(0);
#pragma unroll 1
        for (int c = 0; c < NC; ++c) {
            const int t0 = c * kC, L = min(kC, T - t0), mref = (L - 1) / 2;
            const int par = c & 1;
            wait(MB_RAW, c);
            // ---------------- prefix sums (log2 units), range check, G_m and G_L
            int bad = 0;
            if (SCALAR_G) {
                if (pw == 0) {
                    float *Gp = reinterpret_cast<float *>(smem + kGsc);
                    const float a = gs0 * kLog2e, a2 = gs1 * kLog2e;
                    const float pair = a + a2;
                    float x = pair;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const float yv = __shfl_up_sync(0xffffffffu, x, o);
                        if (lane >= o) x += yv;
                    }
                    const float g_even = x - pair + a;
                    Gp[2 * lane] = g_even;
                    Gp[2 * lane + 1] = x;
                    const float g0 = __shfl_sync(0xffffffffu, g_even, 0);
                    const float gm_e = __shfl_sync(0xffffffffu, g_even, mref >> 1);
                    const float gm_o = __shfl_sync(0xffffffffu, x, mref >> 1);
                    const float gl_e = __shfl_sync(0xffffffffu, g_even, (L - 1) >> 1);
                    const float gl_o = __shfl_sync(0xffffffffu, x, (L - 1) >> 1);
                    const float gmv = (mref & 1) ? gm_o : gm_e;
                    const float glv = ((L - 1) & 1) ? gl_o : gl_e;
                    // each span around the reference row within the half-chunk limit
                    bad = lane == 0 && (g0 - gmv > kHalfLog2 || gmv - glv > kHalfLog2);
                    *reinterpret_cast<float4 *>(vec(kGm, par) + 4 * lane) = make_float4(gmv, gmv, gmv, gmv);
                    *reinterpret_cast<float4 *>(vec(kGL, par) + 4 * lane) = make_float4(glv, glv, glv, glv);
                    load_gsc(t0 + kC);  // the next chunk's log-decays
                }
            } else {
                // warp pw: rows 8 pw .. 8 pw + 7; lane: channels 4 lane .. 4 lane + 3
                float4 x[8];
#pragma unroll
                for (int rr = 0; rr < 8; ++rr) {
                    const float4 v = *reinterpret_cast<const float4 *>(smem + kG + g_off(8 * pw + rr, 4 * lane));
                    const float2 lo = __fmul2_rn(make_float2(v.x, v.y), make_float2(kLog2e, kLog2e));
                    const float2 hi = __fmul2_rn(make_float2(v.z, v.w), make_float2(kLog2e, kLog2e));
                    x[rr] = make_float4(lo.x, lo.y, hi.x, hi.y);
                }
#pragma unroll
                for (int rr = 1; rr < 8; ++rr) {
                    const float2 lo = __fadd2_rn(make_float2(x[rr].x, x[rr].y), make_float2(x[rr - 1].x, x[rr - 1].y));
                    const float2 hi = __fadd2_rn(make_float2(x[rr].z, x[rr].w), make_float2(x[rr - 1].z, x[rr - 1].w));
                    x[rr] = make_float4(lo.x, lo.y, hi.x, hi.y);
                }
                float4 *tot = reinterpret_cast<float4 *>(smem + kTot);
                tot[32 * pw + lane] = x[7];
                named_sync(kNbPrep, kPrepThreads);
                // carry from the blocks above; quarter (blocks 2q, 2q+1) and
                // half (blocks 4h .. 4h+3) decays, each checked once
                float4 carry = make_float4(0.f, 0.f, 0.f, 0.f), half = carry;
#pragma unroll
                for (int w2 = 0; w2 < 7; ++w2) {
                    if (w2 < pw) {
                        const float4 t = tot[32 * w2 + lane];
                        carry = make_float4(carry.x + t.x, carry.y + t.y, carry.z + t.z, carry.w + t.w);
                        if ((w2 >> 2) == (pw >> 2))
                            half = make_float4(half.x + t.x, half.y + t.y, half.z + t.z, half.w + t.w);
                    }
                }
                const float4 own = x[7];
                if (pw & 1) {
                    const float4 t = tot[32 * (pw - 1) + lane];
                    const float q0 = t.x + own.x, q1 = t.y + own.y, q2 = t.z + own.z, q3 = t.w + own.w;
                    bad |= fminf(fminf(q0, q1), fminf(q2, q3)) < -kQuarterLog2;
                }
                if ((pw & 3) == 3) {
                    const float h0v = half.x + own.x, h1v = half.y + own.y, h2v = half.z + own.z,
                                h3v = half.w + own.w;
                    bad |= fminf(fminf(h0v, h1v), fminf(h2v, h3v)) < -kHalfLog2;
                }
#pragma unroll
                for (int rr = 0; rr < 8; ++rr) {
                    const float2 lo = __fadd2_rn(make_float2(x[rr].x, x[rr].y), make_float2(carry.x, carry.y));
                    const float2 hi = __fadd2_rn(make_float2(x[rr].z, x[rr].w), make_float2(carry.z, carry.w));
                    x[rr] = make_float4(lo.x, lo.y, hi.x, hi.y);
                    *reinterpret_cast<float4 *>(smem + kG + g_off(8 * pw + rr, 4 * lane)) = x[rr];
                    // G at the reference row and at the last row
                    if (8 * pw + rr == mref) reinterpret_cast<float4 *>(vec(kGm, par))[lane] = x[rr];
                    if (8 * pw + rr == L - 1) reinterpret_cast<float4 *>(vec(kGL, par))[lane] = x[rr];
                }
            }
            const bool slow = named_sync_or(kNbPrep, kPrepThreads, bad) != 0;
            // ---------------- carry factors: c of the previous chunk, a of this one;
            // after the last chunk, the factor that leaves the final state
            if (pt < kD) {
                const int i = pt;
                const float gm = slow ? 0.f : vec(kGm, par)[i], gl = vec(kGL, par)[i];
                const float a_now = slow ? fast_exp2(gl) : 1.f;
                if (c == 0) {
                    vec(kCv, 1)[i] = fast_exp2(gm);
                    vec(kAv, 1)[i] = a_now;
                } else {
                    const bool sp = slow_flag[par ^ 1] != 0;
                    const float rel = sp ? 0.f : vec(kGL, par ^ 1)[i] - vec(kGm, par ^ 1)[i];
                    vec(kCv, par ^ 1)[i] = fast_exp2(gm + rel);
                    vec(kAv, par ^ 1)[i] = a_now;
                }
            }
            // the prefix sums and carry factors above touch nothing the chain still
            // reads; from here on the Lq, Lk tiles, R of chunk c - 2 and the carry
            // slot of chunk c - 2 are rewritten, all free once chunk c - 1's O^T
            // product (issued after chunk c - 2's state went back to TMEM) is done
            if (c > 0) wait(MB_OPART, c - 1);
            if (c + 1 == NC && pt < kD) {
                const float gm = slow ? 0.f : vec(kGm, par)[pt], gl = vec(kGL, par)[pt];
                vec(kCv, par)[pt] = slow ? 1.f : fast_exp2(gl - gm);
                vec(kAv, par)[pt] = 1.f;
            }
            // ---------------- operand tiles Lq, Lk, R (bf16, K-major core matrices)
            {
                // lane: channel group cg (8 channels) of four, row r8 of eight
                const int cg = 4 * (pw & 3) + (lane >> 3), r8 = lane & 7, ch = 8 * cg;
                float gm[8], gl[8];
                {
                    const float4 m0 = *reinterpret_cast<const float4 *>(vec(kGm, par) + ch);
                    const float4 m1 = *reinterpret_cast<const float4 *>(vec(kGm, par) + ch + 4);
                    const float4 l0 = *reinterpret_cast<const float4 *>(vec(kGL, par) + ch);
                    const float4 l1 = *reinterpret_cast<const float4 *>(vec(kGL, par) + ch + 4);
                    gm[0] = m0.x; gm[1] = m0.y; gm[2] = m0.z; gm[3] = m0.w;
                    gm[4] = m1.x; gm[5] = m1.y; gm[6] = m1.z; gm[7] = m1.w;
                    gl[0] = l0.x; gl[1] = l0.y; gl[2] = l0.z; gl[3] = l0.w;
                    gl[4] = l1.x; gl[5] = l1.y; gl[6] = l1.z; gl[7] = l1.w;
                }
                unsigned char *rbuf = smem + kOpR + par * 16384;
#pragma unroll 2
                for (int kk = 0; kk < 4; ++kk) {
                    const int r = r8 + 8 * (4 * (pw >> 2) + kk);
                    float kv[8], qv[8], gv[8];
                    unpack_bf16x8(*reinterpret_cast<const uint4 *>(smem + kRawK + kq_off(r, ch)), kv);
                    unpack_bf16x8(*reinterpret_cast<const uint4 *>(smem + kRawQ + kq_off(r, ch)), qv);
                    if (SCALAR_G) {
                        const float gr = reinterpret_cast<const float *>(smem + kGsc)[r];
#pragma unroll
                        for (int e = 0; e < 8; ++e) gv[e] = gr;
                    } else {
                        const float4 g0 = *reinterpret_cast<const float4 *>(smem + kG + g_off(r, ch));
                        const float4 g1 = *reinterpret_cast<const float4 *>(smem + kG + g_off(r, ch + 4));
                        gv[0] = g0.x; gv[1] = g0.y; gv[2] = g0.z; gv[3] = g0.w;
                        gv[4] = g1.x; gv[5] = g1.y; gv[6] = g1.z; gv[7] = g1.w;
                    }
                    float lk[8], lq[8], rv[8];
                    if (!slow) {
                        if (SCALAR_G) {  // one decay per row: two exponentials for 8 channels
                            const float d = gv[0] - gm[0];
                            const float el = fast_exp2(d), er = fast_exp2(-d);
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                lk[e] = kv[e] * el;
                                lq[e] = qv[e] * el;
                                rv[e] = kv[e] * er;
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; e += 2) {  // packed fp32 pairs
                                const float2 d = __fadd2_rn(make_float2(gv[e], gv[e + 1]),
                                                            make_float2(-gm[e], -gm[e + 1]));
                                const float2 el = make_float2(fast_exp2(d.x), fast_exp2(d.y));
                                const float2 er = make_float2(fast_exp2(-d.x), fast_exp2(-d.y));
                                const float2 kk2 = make_float2(kv[e], kv[e + 1]);
                                const float2 a = __fmul2_rn(kk2, el);
                                const float2 bq = __fmul2_rn(make_float2(qv[e], qv[e + 1]), el);
                                const float2 cr = __fmul2_rn(kk2, er);
                                lk[e] = a.x; lk[e + 1] = a.y;
                                lq[e] = bq.x; lq[e + 1] = bq.y;
                                rv[e] = cr.x; rv[e + 1] = cr.y;
                            }
                        }
                    } else {
                        // reference row = chunk start: every factor <= 1
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float el = fast_exp2(gv[e]);
                            lk[e] = kv[e] * el;
                            lq[e] = qv[e] * el;
                            rv[e] = kv[e] * fast_exp2(gl[e] - gv[e]);
                        }
                    }
                    *reinterpret_cast<uint4 *>(smem + kOpL + kmajor_off(r, ch, kD)) = pack_bf16x8(lq);
                    *reinterpret_cast<uint4 *>(smem + kOpL + kmajor_off(64 + r, ch, kD)) = pack_bf16x8(lk);
                    *reinterpret_cast<uint4 *>(rbuf + kmajor_off(r, ch, kD)) = pack_bf16x8(rv);
                }
            }
            if (slow) {
                // ---------------- exact path: A (f32, beta-scaled) and P (bf16) block by
                // block, each decay split about a reference row inside the chunk; the
                // solvers must be done with A, and the output product with P
                if (c > 0) {
                    wait(MB_GFREE, c - 1);
                    wait(MB_X, c - 1);
                }
                float *sA = reinterpret_cast<float *>(smem + kA32);
                int *fallback = reinterpret_cast<int *>(smem + kTot);  // [4] diagonal blocks
                // P above the diagonal blocks: zero
                if (pt < 192) {
                    const int u = pt >> 5, I = u < 3 ? 0 : (u < 5 ? 1 : 2);
                    const int J = u < 3 ? u + 1 : (u < 5 ? u - 1 : 3);
                    *reinterpret_cast<uint4 *>(smem + kOpP +
                                               kmajor_off(16 * I + ((pt & 31) >> 1), 16 * J + 8 * (pt & 1), kC)) =
                        make_uint4(0, 0, 0, 0);
                }
                // warp pw: rows 32-47 and 48-63 against columns 0-31 (reference row 32),
                // rows 16-31 against 0-15 (row 16), rows 48-63 against 32-47 (row 48),
                // or diagonal block pw - 4 (its middle row)
                const bool dg = pw >= 4;
                const int r0 = dg ? 16 * (pw - 4) : (pw == 0 ? 32 : (pw == 2 ? 16 : 48));
                const int s0 = dg ? r0 : (pw == 3 ? 32 : 0);
                const int nt_n = pw < 2 ? 4 : 2;
                int b = dg ? r0 + 8 : (pw < 2 ? 32 : r0);
                bool skip = r0 >= L;
                if (dg && !skip) {
                    b = min(b, L - 1);
                    if (!SCALAR_G) {
                        // every factor of the block within range, else pairwise decays
                        const float4 gb4 = *reinterpret_cast<const float4 *>(smem + kG + g_off(b, 4 * lane));
                        float dev = 0.f;
#pragma unroll 4
                        for (int r = r0; r < min(r0 + 16, L); ++r) {
                            const float4 g4 = *reinterpret_cast<const float4 *>(smem + kG + g_off(r, 4 * lane));
                            dev = fmaxf(dev, fmaxf(fmaxf(fabsf(g4.x - gb4.x), fabsf(g4.y - gb4.y)),
                                                   fmaxf(fabsf(g4.z - gb4.z), fabsf(g4.w - gb4.w))));
                        }
                        skip = __any_sync(0xffffffffu, !(dev <= kDiagLog2)) != 0;
                    }
                }
                if (dg && lane == 0) fallback[pw - 4] = (skip && r0 < L) ? 1 : 0;
                const size_t brow = tok0 + t0 + r0 + (lane >> 2);
                const float br0 = r0 + (lane >> 2) < L ? beta[brow * HV + hv] : 0.f;
                const float br1 = r0 + (lane >> 2) + 8 < L ? beta[(brow + 8) * HV + hv] : 0.f;
                exact_block<SCALAR_G>(smem, sA, smem + kOpP, r0, s0, nt_n, b, dg, skip, L, br0, br1, lane);
                named_sync(kNbPrep, kPrepThreads);
                // diagonal blocks out of range: pairwise decays exp(G_r - G_s) <= 1,
                // warp pw on rows pw and pw + 8 of the block, lanes over channels
                __nv_bfloat16 *op = reinterpret_cast<__nv_bfloat16 *>(smem + kOpP);
#pragma unroll 1
                for (int I = 0; I < 4; ++I) {
                    if (!fallback[I]) continue;
#pragma unroll 1
                    for (int r = 16 * I + pw; r < min(16 * I + 16, L); r += 8) {
                        const float br = beta[(tok0 + t0 + r) * HV + hv];
                        const float4 gr4 = *reinterpret_cast<const float4 *>(smem + kG + g_off(r, 4 * lane));
                        const uint2 kr2 = *reinterpret_cast<const uint2 *>(smem + kRawK + kq_off(r, 4 * lane));
                        const uint2 qr2 = *reinterpret_cast<const uint2 *>(smem + kRawQ + kq_off(r, 4 * lane));
                        const float2 k01 = unpack_bf16x2(kr2.x), k23 = unpack_bf16x2(kr2.y);
                        const float2 q01 = unpack_bf16x2(qr2.x), q23 = unpack_bf16x2(qr2.y);
#pragma unroll 1
                        for (int s = 16 * I; s <= r; ++s) {
                            const float4 gs4 = *reinterpret_cast<const float4 *>(smem + kG + g_off(s, 4 * lane));
                            const uint2 ks2 = *reinterpret_cast<const uint2 *>(smem + kRawK + kq_off(s, 4 * lane));
                            const float2 s01 = unpack_bf16x2(ks2.x), s23 = unpack_bf16x2(ks2.y);
                            const float k0 = s01.x * fast_exp2(gr4.x - gs4.x), k1 = s01.y * fast_exp2(gr4.y - gs4.y);
                            const float k2 = s23.x * fast_exp2(gr4.z - gs4.z), k3 = s23.y * fast_exp2(gr4.w - gs4.w);
                            float a = k01.x * k0 + k01.y * k1 + k23.x * k2 + k23.y * k3;
                            float pv = q01.x * k0 + q01.y * k1 + q23.x * k2 + q23.y * k3;
#pragma unroll
                            for (int o = 16; o > 0; o >>= 1) {
                                a += __shfl_xor_sync(0xffffffffu, a, o);
                                pv += __shfl_xor_sync(0xffffffffu, pv, o);
                            }
                            if (lane == 0) {
                                if (s < r) sA[diagT_idx(I, s & 15, r & 15)] = br * a;
                                op[kmajor_off(r, s, kC) >> 1] = __float2bfloat16_rn(pv);
                            }
                        }
                    }
                }
            }
            // the tiles (and on the exact path A and P) are read by the tensor core
            fence_async_smem();
            named_sync(kNbPrep, kPrepThreads);
            if (pt == 0) {
                slow_flag[par] = slow ? 1 : 0;
                mbar_arrive(bar(MB_TILES));
            }
            // ---------------- P read-back (gram rows 0-63): lane quarter 0-1 warps
            if (p_reader) {
                wait(MB_GRAM, c);
                if (!slow) {
                    if (c > 0) wait(MB_X, c - 1);  // the output product has read the previous P
                    tc_fence_after_sync();
                    const int r = 32 * (warp & 3) + lane, s0 = 32 * (pw >> 2);
                    float d[32];
                    tmem_ld32(tl + kTmGram + s0, d);
#pragma unroll
                    for (int u = 0; u < 32; ++u) d[u] = (s0 + u <= r && r < L) ? d[u] : 0.f;
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8)
                        *reinterpret_cast<uint4 *>(smem + kOpP + kmajor_off(r, s0 + 8 * q8, kC)) =
                            pack_bf16x8(&d[8 * q8]);
                    fence_async_smem();
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar(MB_TP));
                    mbar_arrive(bar(MB_GFREE));
                }
            }
        }
    } else if (warp == kWarpChainIssuer) {
        // ================= chain issuer
        const uint32_t vid = idesc_bf16(128, 64, true, false, false);   // V: MN-major A
        const uint32_t ids = idesc_bf16(128, 128, false, true, false);  // R^T: MN-major B
        const uint64_t tdesc = smem_desc(sbase + kOpT, 128, kC * 16);
#pragma unroll 1
        for (int c = 0; c < NC; ++c) {
            named_sync(kNbS, kHandThreads);  // X and S'^T of chunk c are in TMEM
            if (lane == 0) {
                wait(MB_TILES, c);
                if (!*abort_flag) {  // Z^T = S'^T Lk^T
                    tc_fence_after_sync();
                    gemm_ts<kD / 16>(tmem + kTmZ, tmem + kTmSb,
                                     smem_desc(sbase + kOpL + 16384, 128, kD * 16), 256, io, false);
                    mma_commit(bar(MB_Z));
                }
            }
            __syncwarp();
            if (c > 0) named_sync(kNbOfree, kHandThreads);  // O^T of chunk c - 1 is read
            if (lane == 0) {
                if (!*abort_flag) {  // O^T = S'^T Lq^T
                    tc_fence_after_sync();
                    gemm_ts<kD / 16>(tmem + kTmO, tmem + kTmSb, smem_desc(sbase + kOpL, 128, kD * 16),
                                     256, io, false);
                    mma_commit(bar(MB_OPART));
                }
                wait(MB_TP, c);
                wait(MB_V, c);
                if (!*abort_flag) {  // U^T = V^T T'^T (V: 128B-swizzled MN-major)
                    tc_fence_after_sync();
                    gemm_ss<kC / 16>(tmem + kTmU, smem_desc_sw128(sbase + kOpV, 8192, 1024), 2048, tdesc,
                                     256, vid, false);
                }
            }
            __syncwarp();
            named_sync(kNbZb, kHandThreads);
            if (lane == 0 && !*abort_flag) {  // U^T += (-Z^T) T'^T
                tc_fence_after_sync();
                gemm_ts<kC / 16>(tmem + kTmU, tmem + kTmZb, tdesc, 256, io, true);
                mma_commit(bar(MB_U));
            }
            __syncwarp();
            named_sync(kNbUb, kHandThreads);
            if (lane == 0 && !*abort_flag) {
                tc_fence_after_sync();
                // X^T += U^T R (R read transposed), O^T += U^T P^T
                gemm_ts<kC / 16>(tmem + kTmX, tmem + kTmUb,
                                 smem_desc(sbase + kOpR + (c & 1) * 16384, kD * 16, 128), 4096, ids, true);
                gemm_ts<kC / 16>(tmem + kTmO, tmem + kTmUb, smem_desc(sbase + kOpP, 128, kC * 16), 256,
                                 io, true);
                mma_commit(bar(MB_X));
            }
            __syncwarp();
        }
    } else if (warp >= kWarpSolver0) {
        // ================= solver warps: T' of each chunk; warp sw reads the A
        // rows 32 sw .. 32 sw + 31 (TMEM lanes 64 + 32 sw ..)
        const int sw = warp - kWarpSolver0;
        const int st = tid - 32 * kWarpSolver0;  // 0..63
        float *sA = reinterpret_cast<float *>(smem + kA32);
        float *sT = reinterpret_cast<float *>(smem + kT32);
        float *sX = reinterpret_cast<float *>(smem + kX32);
        float *bvec = reinterpret_cast<float *>(smem + kBeta);
        const FragOffsets fo = frag_offsets(lane);
        float bnext = st < T ? beta[(tok0 + st) * HV + hv] : 0.f;
#pragma unroll 1
        for (int c = 0; c < NC; ++c) {
            const int t0 = c * kC, L = min(kC, T - t0);
            bvec[st] = bnext;
            named_sync(kNbSolve, 64);
            if (c + 1 < NC) bnext = t0 + kC + st < T ? beta[(tok0 + t0 + kC + st) * HV + hv] : 0.f;
            wait(MB_GRAM, c);
            if (slow_flag[c & 1] == 0) {
                // A = beta-scaled strictly lower part of gram rows 64-127
                tc_fence_after_sync();
                const int r = 32 * sw + lane, rb = r >> 4;
                const float br = bvec[r];
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    if (sw == 0 && g >= 2) break;  // rows 0-31: column blocks 0-1 only
                    float dd[16];
                    tmem_ld16(tl + kTmGram + 16 * g, dd);
                    if (g == rb) {  // diagonal block, stored transposed
#pragma unroll
                        for (int u = 0; u < 16; ++u)
                            sA[diagT_idx(g, u, r & 15)] = (16 * g + u < r && r < L) ? br * dd[u] : 0.f;
                    } else if (g < rb) {
#pragma unroll
                        for (int u = 0; u < 16; ++u) sA[sq_idx(r, 16 * g + u)] = r < L ? br * dd[u] : 0.f;
                    }
                }
            }
            if (c > 0) wait(MB_U, c - 1);  // the U product has read the previous T'
            // Each solver warp's diagonal blocks and level-1 block use only the
            // rows it wrote itself (or, on the exact path, rows written before
            // the gram barrier): a warp barrier suffices until level 2.
            __syncwarp();
            {
                // diagonal 16 x 16 blocks of T = (I + A)^-1: one thread per column
                // (block I = st / 16, column jj = st % 16), right-looking
                const int I = st >> 4, jj = st & 15;
                float x[16];
#pragma unroll
                for (int p = 0; p < 16; ++p) x[p] = (p == jj) ? 1.f : 0.f;
#pragma unroll
                for (int s2 = 0; s2 < 15; ++s2) {
                    const float4 *col = reinterpret_cast<const float4 *>(sA + diagT_idx(I, s2, 0));
#pragma unroll
                    for (int g4 = (s2 + 1) >> 2; g4 < 4; ++g4) {
                        const float4 a = col[g4];
                        const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (4 * g4 + e > s2) x[4 * g4 + e] = fmaf(-av[e], x[s2], x[4 * g4 + e]);
                    }
                }
                __nv_bfloat16 *opt = reinterpret_cast<__nv_bfloat16 *>(smem + kOpT);
                const float bj = bvec[16 * I + jj];
#pragma unroll
                for (int p = 0; p < 16; p += 2) {
                    sT[sq_idx(16 * I + p, 16 * I + jj)] = x[p];
                    sT[sq_idx(16 * I + p + 1, 16 * I + jj)] = x[p + 1];
                    const __nv_bfloat162 h = __floats2bfloat162_rn(x[p] * bj, x[p + 1] * bj);
                    opt[kmajor_off(16 * I + p, 16 * I + jj, kC) >> 1] = h.x;
                    opt[kmajor_off(16 * I + p + 1, 16 * I + jj, kC) >> 1] = h.y;
                }
            }
            __syncwarp();
            // off-diagonal blocks by 32 x 32 block recursion:
            //   T_10 = -T_11 A_10 T_00,  T_32 = -T_33 A_32 T_22,
            //   [T_20 T_21; T_30 T_31] = -[T_22 0; T_32 T_33] [A_20 A_21; A_30 A_31] [T_00 0; T_10 T_11]
            auto emit = [&](int I, int J, const float (&acc)[2][4]) {  // T_IJ = -acc
                const int gq = lane >> 2, tq = lane & 3;
                float *trow = sT + I * 1024 + 16 * (J ^ (I & 1)) + gq * 64;
                const int u0 = (2 * tq) ^ gq, u1 = (2 * tq + 1) ^ gq;
                unsigned char *prow = smem + kOpT + 2 * I * 1024 + gq * 16 + 4 * tq;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const float2 bb = *reinterpret_cast<const float2 *>(bvec + 16 * J + 8 * nt + 2 * tq);
                    trow[8 * nt + u0] = -acc[nt][0];
                    trow[8 * nt + u1] = -acc[nt][1];
                    trow[512 + 8 * (nt ^ 1) + u0] = -acc[nt][2];
                    trow[512 + 8 * (nt ^ 1) + u1] = -acc[nt][3];
                    // T' = T diag(beta), bf16, K-major [64 r][64 s]
                    *reinterpret_cast<uint32_t *>(prow + (2 * J + nt) * 128) =
                        pack_bf16x2(-acc[nt][0] * bb.x, -acc[nt][1] * bb.y);
                    *reinterpret_cast<uint32_t *>(prow + 1024 + (2 * J + nt) * 128) =
                        pack_bf16x2(-acc[nt][2] * bb.x, -acc[nt][3] * bb.y);
                }
            };
            {  // level 1: block (1,0) on solver 0, (3,2) on solver 1
                const int I = 2 * sw + 1, J = 2 * sw;
                float acc[2][4] = {};
                blk_mma2<true>(acc, swz_block(sA, I, J), swz_block(sT, J, J), fo);
                blk_store(sX + 256 * sw, acc, lane);
                __syncwarp();
                float yv[2][4] = {};
                blk_mma2<false>(yv, swz_block(sT, I, I), sX + 256 * sw, fo);
                emit(I, J, yv);
            }
            named_sync(kNbSolve, 64);
            {  // level 2, row I = 2 + sw of X = [A_20 A_21; A_30 A_31] T1
                const int I = 2 + sw;
                float x0[2][4] = {}, x1[2][4] = {};
                blk_mma2<true>(x0, swz_block(sA, I, 0), swz_block(sT, 0, 0), fo);
                blk_mma2<true>(x0, swz_block(sA, I, 1), swz_block(sT, 1, 0), fo);
                blk_mma2<true>(x1, swz_block(sA, I, 1), swz_block(sT, 1, 1), fo);
                blk_store(sX + 256 * (2 * sw), x0, lane);
                blk_store(sX + 256 * (2 * sw + 1), x1, lane);
            }
            named_sync(kNbSolve, 64);
            {  // level 2, column J = sw of T_lo = -T2 X
                const int J = sw;
                float t2[2][4] = {}, t3[2][4] = {};
                blk_mma2<false>(t2, swz_block(sT, 2, 2), sX + 256 * J, fo);
                blk_mma2<false>(t3, swz_block(sT, 3, 2), sX + 256 * J, fo);
                blk_mma2<false>(t3, swz_block(sT, 3, 3), sX + 256 * (2 + J), fo);
                emit(2, J, t2);
                emit(3, J, t3);
            }
            fence_async_smem();  // T' is read by the tensor core
            tc_fence_before_sync();
            named_sync(kNbSolve, 64);
            if (st == 0) {
                mbar_arrive(bar(MB_TP));
                mbar_arrive(bar(MB_GFREE));
            }
        }
    } else {
        // ================= producer (lane 0).  Per chunk c: once chunk c's
        // tiles are built, the raw k, q, g copies of chunk c + 1 (their buffers
        // are free) and the gram of chunk c (once the previous gram is read);
        // then v of chunk c (once chunk c - 1's U product has read v).
        if (lane == 0) {
            if (VARLEN) {
                // the maps were written to global memory before the launch
                fence_tensormap_acquire(&m.k);
                fence_tensormap_acquire(&m.q);
                if (!SCALAR_G) fence_tensormap_acquire(&m.g);
                fence_tensormap_acquire(&m.v);
            }
            tma_prefetch_desc(&m.k);
            tma_prefetch_desc(&m.q);
            if (!SCALAR_G) tma_prefetch_desc(&m.g);
            tma_prefetch_desc(&m.v);
            auto load_raw = [&](int t0) {
                if (*abort_flag) return;
                mbar_arrive_expect_tx(bar(MB_RAW), SCALAR_G ? kBytesKQG - 32768 : kBytesKQG);
                tma_load_4d(smem + kRawK, &m.k, 0, hk, t0, b, bar(MB_RAW));
                tma_load_4d(smem + kRawK + 8192, &m.k, 64, hk, t0, b, bar(MB_RAW));
                tma_load_4d(smem + kRawQ, &m.q, 0, hk, t0, b, bar(MB_RAW));
                tma_load_4d(smem + kRawQ + 8192, &m.q, 64, hk, t0, b, bar(MB_RAW));
                if (!SCALAR_G) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        tma_load_4d(smem + kG + 8192 * q4, &m.g, 32 * q4, hv, t0, b, bar(MB_RAW));
                }
                ++issued_raw;
            };
            load_raw(0);
#pragma unroll 1
            for (int c = 0; c < NC; ++c) {
                wait(MB_TILES, c);
                if (c + 1 < NC) load_raw((c + 1) * kC);
                if (c > 0) wait(MB_GFREE, c - 1);
                if (slow_flag[c & 1] != 0) {
                    mbar_arrive(bar(MB_GRAM));  // A and P came from the exact path
                } else if (!*abort_flag) {
                    tc_fence_after_sync();
                    gemm_ss<kD / 16>(tmem + kTmGram, smem_desc(sbase + kOpL, 128, kD * 16), 256,
                                     smem_desc(sbase + kOpR + (c & 1) * 16384, 128, kD * 16), 256, io,
                                     false);
                    mma_commit(bar(MB_GRAM));
                }
                if (c > 0) wait(MB_U, c - 1);
                if (!*abort_flag) {
                    mbar_arrive_expect_tx(bar(MB_V), kBytesV);
                    tma_load_4d(smem + kOpV, &m.v, 0, hv, c * kC, b, bar(MB_V));
                    tma_load_4d(smem + kOpV + 8192, &m.v, 64, hv, c * kC, b, bar(MB_V));
                    ++issued_v;
                }
            }
        }
        __syncwarp();
    }

    __syncthreads();
    const bool aborted = *abort_flag != 0;
    if (tid == 0 && aborted) atomicOr(dev_error, 1);
    if (warp == kWarpProducer && lane == 0 && aborted) {
        // never leave with copies in flight: wait (bounded) for the last copy
        // issued on each barrier; its phases complete in order
        if (issued_raw > 0) mbar_wait_bounded(bar(MB_RAW), (uint32_t)((issued_raw - 1) & 1), kWaitLimitNs);
        if (issued_v > 0) mbar_wait_bounded(bar(MB_V), (uint32_t)((issued_v - 1) & 1), kWaitLimitNs);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// The five tensor maps of a [B][T][H][128] problem whose token 0 of batch 0
// sits at row `tok0` of the packed tensors.
bool encode_maps(EncodeTiledFn fn, TileMaps *tm, const Problem &p, size_t tok0, int B, int T) {
    const char *q = static_cast<const char *>(p.q) + tok0 * p.HK * kD * 2;
    const char *k = static_cast<const char *>(p.k) + tok0 * p.HK * kD * 2;
    const char *v = static_cast<const char *>(p.v) + tok0 * p.HV * kD * 2;
    const char *g = reinterpret_cast<const char *>(p.g) + tok0 * p.HV * kD * 4;
    const char *o = static_cast<const char *>(p.out) + tok0 * p.HV * kD * 2;
    // a scalar gate's g is read without a tensor map
    if (p.g_scalar) memset(&tm->g, 0, sizeof(tm->g));
    const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
    return tma_encode_rows(fn, &tm->k, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, T, p.HK, 64, sw, 64) &&
           tma_encode_rows(fn, &tm->q, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, T, p.HK, 64, sw, 64) &&
           (p.g_scalar ||
            tma_encode_rows(fn, &tm->g, g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, B, T, p.HV, 32, sw, 64)) &&
           tma_encode_rows(fn, &tm->v, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, T, p.HV, 64, sw, 64) &&
           // output: unswizzled [32 tokens][32 channels] boxes, one per chain warp
           tma_encode_rows(fn, &tm->o, o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, T, p.HV, 32,
                           CU_TENSOR_MAP_SWIZZLE_NONE, 32);
}

template <bool VARLEN, bool SCALAR_G>
cudaError_t launch_tc(const Problem &p, const TileMaps &tm, const TileMaps *seq_maps,
                      const int4 *seqs, long long blocks, int *dev_error, cudaStream_t stream) {
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (blocks == 0) return cudaSuccess;
    auto run = [&](auto kernel) -> cudaError_t {
        cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)kSmemBytes);
        if (err != cudaSuccess) return err;
        trace_begin(kKernFused, stream);
        kernel<<<(unsigned)blocks, kThreads, kSmemBytes, stream>>>(
            tm, seq_maps, seqs, p.beta, p.g, p.h0, p.ht, p.T, p.HK, p.HV, dev_error);
        trace_end(kKernFused, stream);
        return cudaGetLastError();
    };
    if (p.h0 && p.ht) return run(gdr_prefill_tc_kernel<true, true, VARLEN, SCALAR_G>);
    if (p.h0) return run(gdr_prefill_tc_kernel<true, false, VARLEN, SCALAR_G>);
    if (p.ht) return run(gdr_prefill_tc_kernel<false, true, VARLEN, SCALAR_G>);
    return run(gdr_prefill_tc_kernel<false, false, VARLEN, SCALAR_G>);
}

}  // namespace

bool tc_prefill_supported(const Problem &p) {
    return p.bf16 && p.dk == kD && p.dv == kD && p.chunk == kC;
}

cudaError_t launch_tc_prefill(const Problem &p, int *dev_error, cudaStream_t stream) {
    cudaError_t e = cudaSuccess;
    EncodeTiledFn fn = tma_encode_fn(&e);
    if (e != cudaSuccess) return e;
    TileMaps tm;
    if (!encode_maps(fn, &tm, p, 0, p.B, p.T)) return cudaErrorInvalidValue;
    const long long blocks = (long long)p.B * p.HV;
    return p.g_scalar ? launch_tc<false, true>(p, tm, nullptr, nullptr, blocks, dev_error, stream)
                      : launch_tc<false, false>(p, tm, nullptr, nullptr, blocks, dev_error, stream);
}

size_t tc_seq_maps_bytes() { return sizeof(TileMaps); }

cudaError_t tc_encode_seq_maps(const Problem &p, size_t tok0, int L, void *dst,
                               const void *v_row, void *o_row) {
    cudaError_t e = cudaSuccess;
    EncodeTiledFn fn = tma_encode_fn(&e);
    if (e != cudaSuccess) return e;
    TileMaps tm;
    if (!encode_maps(fn, &tm, p, tok0, 1, L)) return cudaErrorInvalidValue;
    // one-row stand-ins: every load past row 0 reads the zero fill, every
    // store past row 0 is dropped
    if (v_row && !tma_encode_rows(fn, &tm.v, v_row, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 1, 1, p.HV,
                                  64, CU_TENSOR_MAP_SWIZZLE_128B, 64))
        return cudaErrorInvalidValue;
    if (o_row && !tma_encode_rows(fn, &tm.o, o_row, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 1, 1, p.HV,
                                  32, CU_TENSOR_MAP_SWIZZLE_NONE, 32))
        return cudaErrorInvalidValue;
    memcpy(dst, &tm, sizeof(TileMaps));
    return cudaSuccess;
}

cudaError_t launch_tc_prefill_varlen(const Problem &p, const void *seq_maps, const int4 *seqs,
                                     int nseq, int *dev_error, cudaStream_t stream) {
    TileMaps unused;
    memset(&unused, 0, sizeof(unused));
    const TileMaps *maps = static_cast<const TileMaps *>(seq_maps);
    return p.g_scalar
               ? launch_tc<true, true>(p, unused, maps, seqs, (long long)nseq * p.HV, dev_error, stream)
               : launch_tc<true, false>(p, unused, maps, seqs, (long long)nseq * p.HV, dev_error, stream);
}

}  // namespace gdr
