// prefill_tc.cu -- chunkwise WY/UT prefill on the Blackwell tensor cores
// (tcgen05 MMA, TMEM accumulators) for bf16 q/k/v with dk = dv = 128 and
// chunks of 64 tokens, fused into one kernel.
//
// Method: page "Reorder channelwise gated delta rule chunked hot loops for
// autovectorization" (pytorch/executorch PR #21021), second commit summary --
// per chunk: per-channel log-decay prefix sums, the causal query/key terms,
// the beta-folded unit-lower triangular transform, WY pseudo-keys and
// pseudo-values, and the state carried to the next chunk, with a ragged last
// chunk through the same code.  The triangular transform is a block forward
// substitution (16 x 16 diagonal-block inverses, then the off-diagonal blocks
// by small matrix products), the block-TRSM structure of trymirai/uzu PR #576
// ("Support TreeUpdateSolve kernel", commit summary).
//
// Algebra per chunk of L <= 64 tokens (r, s local token indices; S the state
// at the chunk start; G the inclusive per-channel prefix sum of g):
//   A[r,s] = beta_r sum_i k_ri k_si exp(G_ri - G_si)   (s < r)
//   P[r,s] =        sum_i q_ri k_si exp(G_ri - G_si)   (s <= r)
//   T'     = (I + A)^-1 diag(beta)
//   U      = T' V - T' (exp(G) * K) S
//   O      = (exp(G) * Q) S + P U
//   S     <- diag(exp(G_L)) S + (exp(G_L - G) * K)^T U
//
// Factoring around a reference row m of the chunk.  With
//   Lk = K * exp(G - G_m),  Lq = Q * exp(G - G_m),  R = K * exp(G_m - G),
//   S' = diag(exp(G_m)) S,
// every product above is a product of these three tiles:
//   A = tril(diag(beta) Lk R^T),  P = tril(Lq R^T),
//   (exp(G) * K) S = Lk S',  (exp(G) * Q) S = Lq S',
//   (exp(G_L - G) * K)^T U = diag(exp(G_L - G_m)) R^T U.
// While every channel decays by at most 80 nats between the chunk's first
// token and m and between m and its last token, all factors are finite and
// the products are exact to rounding.  A chunk outside that range (decay
// stronger than ~2.5 nats per token sustained over 32 tokens) uses m := the
// chunk start instead (Lk = exp(G) K, Lq = exp(G) Q, R = exp(G_L - G) K, all
// factors <= 1) and computes A and P with exact pairwise decays on CUDA
// cores, so the result is right for any g <= 0.
//
// GB300 mapping.  One CTA (8 warps) per (batch, value head) walks that head's
// chunks in order; the float32 state never leaves registers (thread = one
// value column j, 64 of the 128 key rows).  State products are computed
// transposed so that M = dv = 128 fills the MMA:
//   U^T = (T'V)^T - S'^T (T'Lk)^T,  O^T = S'^T Lq^T + U^T P^T,  dS^T = U^T R.
// Operands are bf16 tiles in shared memory in the interleaved (no-swizzle)
// core-matrix layout (sm100_ptx.cuh); each of Lk, Lq and R is stored once
// and read both K-major and, through an MN-major descriptor with the two
// core-matrix strides exchanged, transposed.  Accumulators are float32 in
// TMEM.  The next chunk's inputs are fetched with cp.async while the current
// chunk's solve and state products run.  The 64 x 64 inverse runs in
// float32: diagonal blocks by a right-looking sweep per column, off-diagonal
// blocks by tf32 mma.sync 16 x 16 products.
#include "common.cuh"
#include "sm100_ptx.cuh"

namespace gdr {
namespace {

using namespace sm100;

constexpr int kC = 64;      // chunk length
constexpr int kD = 128;     // dk = dv
constexpr int kThreads = 256;
constexpr float kRangeNats = 80.f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per MMA batch

// ---- shared memory map (bytes)
constexpr uint32_t kRawK = 0;                 // bf16 [64][128], 16-byte chunks XOR-swizzled by row
constexpr uint32_t kRawQ = kRawK + 16384;     // same for q
constexpr uint32_t kOpV = kRawQ + 16384;      // V as MN-major A (k = s, mn = j), K extent 64
constexpr uint32_t kG = kOpV + 16384;         // f32 [64][128], 16-byte chunks XOR-swizzled by row
constexpr uint32_t kOpL = kG + 32768;         // [128][128] K-major: rows 0-63 Lk, 64-127 Lq
constexpr uint32_t kOpR = kOpL + 32768;       // [64][128] K-major: R
constexpr uint32_t kAT = kOpR + 16384;        // 32 KB: f32 A and T (64x64 each), later S'^T
constexpr uint32_t kA32 = kAT;
constexpr uint32_t kT32 = kAT + 16384;
constexpr uint32_t kOpST = kAT;               //   S'^T as K-major A [128 j][128 i]
constexpr uint32_t kOpT = kAT + 32768;        // T' as K-major B [64 r][64 s]
constexpr uint32_t kOpP = kOpT + 8192;        // P as K-major B [64 r][64 s]
constexpr uint32_t kOpWK = kOpP + 8192;       // (T'Lk) as MN-major B (k = i, mn = r), K extent 128
constexpr uint32_t kStage = kOpWK;            //   later: bf16 O [64][128] staging for the stores
constexpr uint32_t kOpUT = kOpWK + 16384;     // U^T as K-major A [128 j][64 r]
constexpr uint32_t kX32 = kOpUT;              //   earlier: f32 [3][16][16] solve scratch
constexpr uint32_t kSmall = kOpUT + 16384;
constexpr uint32_t kBeta = kSmall;            // f32 [2][64] (double-buffered)
constexpr uint32_t kEGm = kBeta + 512;        // f32 [128] exp(G_m)
constexpr uint32_t kCL = kEGm + 512;          // f32 [128] exp(G_last - G_m)
constexpr uint32_t kGamL = kCL + 512;         // f32 [128] exp(G_last)
constexpr uint32_t kGm = kGamL + 512;         // f32 [128] G_m
constexpr uint32_t kTot = kGm + 512;          // f32 [128] prefix-sum carry
constexpr uint32_t kBar = kTot + 512;         // mbarrier (8 B)
constexpr uint32_t kTmemSlot = kBar + 8;      // u32
constexpr uint32_t kSmemBytes = kTmemSlot + 8;
static_assert(kSmemBytes <= 232448, "shared memory budget");

// ---- TMEM columns (float32 accumulators, lane = M row)
constexpr uint32_t kTmGram = 0;     // [128 x 64]: rows 0-63 Lk R^T, 64-127 Lq R^T
constexpr uint32_t kTmWkT = 64;     // [128 i x 64 r]  (T' Lk)^T
constexpr uint32_t kTmUT = 128;     // [128 j x 64 r]
constexpr uint32_t kTmOT = 192;     // [128 j x 64 r]
constexpr uint32_t kTmDS = 256;     // [128 j x 128 i]
constexpr uint32_t kTmemCols = 512;

// 64 x 64 f32 tiles (A, T) with an XOR swizzle: rows and columns both walk
// conflict-free
__device__ __forceinline__ int sq_idx(int r, int s) { return r * 64 + (s ^ (r & 31)); }
// raw bf16 [64][128]: element offset of (r, i)
__device__ __forceinline__ int rawkq_idx(int r, int i) {
    return r * 128 + ((((i >> 3) ^ (r & 7))) << 3) + (i & 7);
}
// G f32 [64][128]: element offset of (r, i)
__device__ __forceinline__ int g_idx(int r, int i) {
    return r * 128 + ((((i >> 2) ^ (r & 7))) << 2) + (i & 3);
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

// Issues the K-steps of one GEMM, D (+)= A * B^T, each K-step of 16
// advancing the operand start addresses by two core matrices along K.
__device__ __forceinline__ void gemm(uint32_t d_tmem, uint32_t a_addr, uint32_t a_lbo,
                                     uint32_t a_sbo, uint32_t b_addr, uint32_t b_lbo,
                                     uint32_t b_sbo, uint32_t idesc, int k_steps,
                                     bool accumulate_first) {
    for (int ks = 0; ks < k_steps; ++ks) {
        const uint64_t ad = smem_desc(a_addr + ks * 2 * a_lbo, a_lbo, a_sbo);
        const uint64_t bd = smem_desc(b_addr + ks * 2 * b_lbo, b_lbo, b_sbo);
        mma_bf16(d_tmem, ad, bd, idesc, (ks > 0 || accumulate_first) ? 1u : 0u);
    }
}

// Waits for the CTA's MMA batch; false (uniform across the CTA) on timeout.
__device__ __forceinline__ bool wait_mma(uint64_t *bar, uint32_t &phase) {
    const bool ok = mbar_wait_bounded(bar, phase, kWaitLimitNs);
    phase ^= 1u;
    const int any_fail = __syncthreads_or(ok ? 0 : 1);
    tc_fence_after_sync();
    return any_fail == 0;
}

// ---- tf32 mma.sync for the 16 x 16 block products of the inverse
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void mma_tf32(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Issues the cp.async copies of one chunk's k, q, g rows (rows >= L zeroed).
__device__ __forceinline__ void load_kqg(unsigned char *smem, const __nv_bfloat16 *k,
                                         const __nv_bfloat16 *q, const float *g, int b, int T,
                                         int t0, int L, int HK, int HV, int hk, int hv, int tid) {
    const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int id = tid + kThreads * it;  // 0..1023
        const int r = id >> 4, cc = id & 15;
        const int pc = cc ^ (r & 7);
        unsigned char *dk_ = smem + kRawK + r * 256 + pc * 16;
        unsigned char *dq_ = smem + kRawQ + r * 256 + pc * 16;
        if (r < L) {
            const size_t tk = ((size_t)b * T + t0 + r) * HK + hk;
            cp_async16(dk_, k + tk * kD + cc * 8);
            cp_async16(dq_, q + tk * kD + cc * 8);
        } else {
            *reinterpret_cast<uint4 *>(dk_) = zero4;
            *reinterpret_cast<uint4 *>(dq_) = zero4;
        }
    }
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int id = tid + kThreads * it;  // 0..2047
        const int r = id >> 5, cc = id & 31;
        unsigned char *dg = smem + kG + r * 512 + ((cc ^ (r & 7)) * 16);
        if (r < L)
            cp_async16(dg, g + (((size_t)b * T + t0 + r) * HV + hv) * kD + cc * 4);
        else
            *reinterpret_cast<uint4 *>(dg) = zero4;
    }
}
__device__ __forceinline__ void load_v(unsigned char *smem, const __nv_bfloat16 *v, int b, int T,
                                       int t0, int L, int HV, int hv, int tid) {
    const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int id = tid + kThreads * it;
        const int r = id >> 4, cc = id & 15;
        unsigned char *dv_ = smem + kOpV + mnmajor_off(r, cc * 8, kC);
        if (r < L)
            cp_async16(dv_, v + (((size_t)b * T + t0 + r) * HV + hv) * kD + cc * 8);
        else
            *reinterpret_cast<uint4 *>(dv_) = zero4;
    }
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait0() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

template <bool HAS_H0, bool STORE_HT>
__global__ void __launch_bounds__(kThreads, 1)
    gdr_prefill_tc_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                          const __nv_bfloat16 *__restrict__ v, const float *__restrict__ g,
                          const float *__restrict__ beta, const float *h0,
                          __nv_bfloat16 *__restrict__ out, float *ht, int T, int HK, int HV,
                          int *dev_error) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wq = warp & 3;        // TMEM lane quarter of this warp
    const int ih = warp >> 2;       // which half of the key channels / tokens this warp takes
    const int head = blockIdx.x;    // b * HV + hv
    const int hv = head % HV, b = head / HV;
    const int hk = hv / (HV / HK);
    const int j = 32 * wq + lane;   // this thread's value column (TMEM lane)

    float *sEGm = reinterpret_cast<float *>(smem + kEGm);
    float *sCL = reinterpret_cast<float *>(smem + kCL);
    float *sGamL = reinterpret_cast<float *>(smem + kGamL);
    float *sGm = reinterpret_cast<float *>(smem + kGm);
    float *sTot = reinterpret_cast<float *>(smem + kTot);
    float *sG = reinterpret_cast<float *>(smem + kG);
    float *sA = reinterpret_cast<float *>(smem + kA32);
    float *sT = reinterpret_cast<float *>(smem + kT32);
    float *sX = reinterpret_cast<float *>(smem + kX32);
    const __nv_bfloat16 *rawk = reinterpret_cast<const __nv_bfloat16 *>(smem + kRawK);
    const __nv_bfloat16 *rawq = reinterpret_cast<const __nv_bfloat16 *>(smem + kRawQ);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kTmemSlot);

    if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    const int NC = (T + kC - 1) / kC;
    // first chunk's inputs
    {
        const int L0 = min(kC, T);
        load_kqg(smem, k, q, g, b, T, 0, L0, HK, HV, hk, hv, tid);
        load_v(smem, v, b, T, 0, L0, HV, hv, tid);
        cp_async_commit();
        float *sb0 = reinterpret_cast<float *>(smem + kBeta);
        if (tid < kC) sb0[tid] = tid < L0 ? beta[((size_t)b * T + tid) * HV + hv] : 0.f;
    }
    // state: S[64*ih + u][j], u = 0..63
    float S[64];
#pragma unroll
    for (int u = 0; u < 64; ++u)
        S[u] = HAS_H0 ? h0[((size_t)head * kD + 64 * ih + u) * kD + j] : 0.f;
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tl = tmem + ((uint32_t)(32 * wq) << 16);  // this warp's lane quarter
    uint32_t phase = 0;
    bool aborted = false;

    for (int c = 0; c < NC; ++c) {
        const int t0 = c * kC;
        const int L = min(kC, T - t0);
        const int m = (L - 1) / 2;  // reference row of the factorisation
        const float *sbeta = reinterpret_cast<const float *>(smem + kBeta + 256 * (c & 1));
        const bool has_next = c + 1 < NC;
        const int t0n = t0 + kC;
        const int Ln = has_next ? min(kC, T - t0n) : 0;

        cp_async_wait0();
        __syncthreads();

        // ---------------- per-channel prefix sums of g (two halves of 32 rows)
        {
            const int i = tid & 127, hh = tid >> 7;
            float x[32];
#pragma unroll
            for (int r = 0; r < 32; ++r) x[r] = sG[g_idx(32 * hh + r, i)];
#pragma unroll
            for (int r = 1; r < 32; ++r) x[r] += x[r - 1];
            if (hh == 0) sTot[i] = x[31];
            __syncthreads();
            if (hh == 1) {
                const float carry = sTot[i];
#pragma unroll
                for (int r = 0; r < 32; ++r) x[r] += carry;
            }
#pragma unroll
            for (int r = 0; r < 32; ++r) sG[g_idx(32 * hh + r, i)] = x[r];
        }
        __syncthreads();
        int bad = 0;
        if (tid < kD) {
            const int i = tid;
            const float g0 = sG[g_idx(0, i)], gm = sG[g_idx(m, i)], gl = sG[g_idx(L - 1, i)];
            bad = (g0 - gm > kRangeNats) || (gm - gl > kRangeNats);
            sGm[i] = gm;
            sGamL[i] = __expf(gl);
        }
        const bool slow = __syncthreads_or(bad) != 0;
        if (tid < kD) {
            // the fallback factorises around the chunk start (G_m = 0) and
            // stores R with the full decay to the chunk end (scale 1)
            const float gm = slow ? 0.f : sGm[tid];
            sGm[tid] = gm;
            sEGm[tid] = slow ? 1.f : __expf(gm);
            sCL[tid] = slow ? 1.f : __expf(sG[g_idx(L - 1, tid)] - gm);
        }
        __syncthreads();

        // ---------------- operands Lk, Lq, R (bf16, K-major core-matrix tiles)
#pragma unroll 2
        for (int it = 0; it < 4; ++it) {
            const int id = tid + kThreads * it;  // 0..1023
            const int r8 = id & 7;
            const int r = ((id >> 7) << 3) | r8;
            const int c8 = (id >> 3) & 15;
            const int ch = c8 * 8;
            float kv[8], qv[8];
            unpack_bf16x8(*reinterpret_cast<const uint4 *>(smem + kRawK + r * 256 + ((c8 ^ r8) << 4)), kv);
            unpack_bf16x8(*reinterpret_cast<const uint4 *>(smem + kRawQ + r * 256 + ((c8 ^ r8) << 4)), qv);
            const float4 g_lo = *reinterpret_cast<const float4 *>(smem + kG + r * 512 + (((2 * c8) ^ r8) << 4));
            const float4 g_hi = *reinterpret_cast<const float4 *>(smem + kG + r * 512 + (((2 * c8 + 1) ^ r8) << 4));
            const float4 m_lo = *reinterpret_cast<const float4 *>(sGm + ch);
            const float4 m_hi = *reinterpret_cast<const float4 *>(sGm + ch + 4);
            const float d[8] = {g_lo.x - m_lo.x, g_lo.y - m_lo.y, g_lo.z - m_lo.z, g_lo.w - m_lo.w,
                                g_hi.x - m_hi.x, g_hi.y - m_hi.y, g_hi.z - m_hi.z, g_hi.w - m_hi.w};
            float lk[8], lq[8], rk[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float el = __expf(d[e]);
                lk[e] = kv[e] * el;
                lq[e] = qv[e] * el;
            }
            if (!slow) {
#pragma unroll
                for (int e = 0; e < 8; ++e) rk[e] = kv[e] * __expf(-d[e]);
            } else {
                // G_m = 0 here, so d = G; R = exp(G_L - G) K directly (factor <= 1)
#pragma unroll
                for (int e = 0; e < 8; ++e) rk[e] = kv[e] * __expf(sG[g_idx(L - 1, ch + e)] - d[e]);
            }
            *reinterpret_cast<uint4 *>(smem + kOpL + kmajor_off(r, ch, kD)) = pack_bf16x8(lk);
            *reinterpret_cast<uint4 *>(smem + kOpL + kmajor_off(64 + r, ch, kD)) = pack_bf16x8(lq);
            *reinterpret_cast<uint4 *>(smem + kOpR + kmajor_off(r, ch, kD)) = pack_bf16x8(rk);
        }
        fence_async_smem();
        __syncthreads();

        // ---------------- MMA batch 1: gram [Lk; Lq] R^T
        if (!slow) {
            if (tid == 0) {
                tc_fence_after_sync();
                gemm(tmem + kTmGram, sbase + kOpL, 128, kD * 16, sbase + kOpR, 128, kD * 16,
                     idesc_bf16(128, 64, false, false, false), kD / 16, false);
                mma_commit(bar);
            }
            if (!wait_mma(bar, phase)) { aborted = true; break; }
            // A (f32, beta-folded, strictly lower) and P (bf16, causal)
            float dd[32];
            tmem_ld32(tl + kTmGram + 32 * ih, dd);
            const int row = 32 * wq + lane;
            if (row < kC) {
                const int r = row;
                const float br = sbeta[r];
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    const int s = 32 * ih + u;
                    sA[sq_idx(r, s)] = (s < r && r < L) ? br * dd[u] : 0.f;
                }
            } else {
                const int r = row - kC;
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    const int s = 32 * ih + u;
                    dd[u] = (s <= r && r < L) ? dd[u] : 0.f;
                }
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8)
                    *reinterpret_cast<uint4 *>(smem + kOpP + kmajor_off(r, 32 * ih + 8 * q8, kC)) =
                        pack_bf16x8(&dd[8 * q8]);
            }
        } else {
            // exact pairwise decays on CUDA cores (every exponent <= 0)
            __nv_bfloat16 *op = reinterpret_cast<__nv_bfloat16 *>(smem + kOpP);
            for (int idx = tid; idx < kC * kC; idx += kThreads) {
                const int r = idx >> 6, s = idx & 63;
                float a = 0.f, p = 0.f;
                if (s <= r && r < L) {
                    for (int i = 0; i < kD; ++i) {
                        const float e = __expf(sG[g_idx(r, i)] - sG[g_idx(s, i)]);
                        const float kse = __bfloat162float(rawk[rawkq_idx(s, i)]) * e;
                        a = fmaf(__bfloat162float(rawk[rawkq_idx(r, i)]), kse, a);
                        p = fmaf(__bfloat162float(rawq[rawkq_idx(r, i)]), kse, p);
                    }
                }
                sA[sq_idx(r, s)] = (s < r) ? sbeta[r] * a : 0.f;
                op[kmajor_off(r, s, kC) >> 1] = __float2bfloat16_rn(p);
            }
        }
        tc_fence_before_sync();
        __syncthreads();

        // prefetch the next chunk's k, q, g (their buffers are free now)
        if (has_next) {
            load_kqg(smem, k, q, g, b, T, t0n, Ln, HK, HV, hk, hv, tid);
            cp_async_commit();
            float *sbn = reinterpret_cast<float *>(smem + kBeta + 256 * ((c + 1) & 1));
            if (tid < kC) sbn[tid] = tid < Ln ? beta[((size_t)b * T + t0n + tid) * HV + hv] : 0.f;
        }

        // ---------------- T = (I + A)^-1, diagonal 16 x 16 blocks (right-looking)
        if (tid < 64) {
            const int I = tid >> 4, jj = tid & 15;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) x[r] = (r == jj) ? 1.f : 0.f;
#pragma unroll
            for (int s = 0; s < 15; ++s) {
#pragma unroll
                for (int r = s + 1; r < 16; ++r)
                    x[r] = fmaf(-sA[sq_idx(16 * I + r, 16 * I + s)], x[s], x[r]);
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) sT[sq_idx(16 * I + r, 16 * I + jj)] = x[r];
        }
        __syncthreads();
        // ---------------- off-diagonal blocks, level by level: T_IJ = -T_II sum_M A_IM T_MJ
        {
            const int gq = lane >> 2, tq = lane & 3;
#pragma unroll 1
            for (int dlev = 1; dlev < 4; ++dlev) {
                if (warp < 4 - dlev) {
                    const int J = warp, I = J + dlev;
                    float xc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                    for (int M = J; M < I; ++M) {
#pragma unroll
                        for (int kh = 0; kh < 2; ++kh) {
                            const int kc = 16 * M + 8 * kh + tq;
                            uint32_t a[4];
                            a[0] = to_tf32(sA[sq_idx(16 * I + gq, kc)]);
                            a[1] = to_tf32(sA[sq_idx(16 * I + gq + 8, kc)]);
                            a[2] = to_tf32(sA[sq_idx(16 * I + gq, kc + 4)]);
                            a[3] = to_tf32(sA[sq_idx(16 * I + gq + 8, kc + 4)]);
#pragma unroll
                            for (int nt = 0; nt < 2; ++nt) {
                                const int n = 16 * J + 8 * nt + gq;
                                mma_tf32(xc[nt], a, to_tf32(sT[sq_idx(kc, n)]),
                                         to_tf32(sT[sq_idx(kc + 4, n)]));
                            }
                        }
                    }
                    float *xs = sX + warp * 256;  // X as f32 [16][16]
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        xs[gq * 16 + 8 * nt + 2 * tq] = xc[nt][0];
                        xs[gq * 16 + 8 * nt + 2 * tq + 1] = xc[nt][1];
                        xs[(gq + 8) * 16 + 8 * nt + 2 * tq] = xc[nt][2];
                        xs[(gq + 8) * 16 + 8 * nt + 2 * tq + 1] = xc[nt][3];
                    }
                    __syncwarp();
                    float yc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                    for (int kh = 0; kh < 2; ++kh) {
                        const int kc = 16 * I + 8 * kh + tq;
                        uint32_t a[4];
                        a[0] = to_tf32(sT[sq_idx(16 * I + gq, kc)]);
                        a[1] = to_tf32(sT[sq_idx(16 * I + gq + 8, kc)]);
                        a[2] = to_tf32(sT[sq_idx(16 * I + gq, kc + 4)]);
                        a[3] = to_tf32(sT[sq_idx(16 * I + gq + 8, kc + 4)]);
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
                            const int kx = 8 * kh + tq, n = 8 * nt + gq;
                            mma_tf32(yc[nt], a, to_tf32(xs[kx * 16 + n]), to_tf32(xs[(kx + 4) * 16 + n]));
                        }
                    }
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const int col = 16 * J + 8 * nt + 2 * tq;
                        sT[sq_idx(16 * I + gq, col)] = -yc[nt][0];
                        sT[sq_idx(16 * I + gq, col + 1)] = -yc[nt][1];
                        sT[sq_idx(16 * I + gq + 8, col)] = -yc[nt][2];
                        sT[sq_idx(16 * I + gq + 8, col + 1)] = -yc[nt][3];
                    }
                }
                __syncthreads();
            }
        }
        // T' = T diag(beta) as bf16 (zero above the diagonal)
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const int id = tid + kThreads * it;  // 0..511
            const int r = id & 63, s0 = (id >> 6) * 8;
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int s = s0 + e;
                x[e] = (s <= r) ? sT[sq_idx(r, s)] * sbeta[s] : 0.f;
            }
            *reinterpret_cast<uint4 *>(smem + kOpT + kmajor_off(r, s0, kC)) = pack_bf16x8(x);
        }
        fence_async_smem();
        __syncthreads();

        // ---------------- MMA batch 2: (T'Lk)^T = Lk^T T'^T,  U^T = V^T T'^T
        if (tid == 0) {
            tc_fence_after_sync();
            // Lk read transposed: MN-major (k = s, mn = i), K-direction stride 2048, MN 128
            gemm(tmem + kTmWkT, sbase + kOpL, kD * 16, 128, sbase + kOpT, 128, kC * 16,
                 idesc_bf16(128, 64, true, false, false), kC / 16, false);
            gemm(tmem + kTmUT, sbase + kOpV, 128, kC * 16, sbase + kOpT, 128, kC * 16,
                 idesc_bf16(128, 64, true, false, false), kC / 16, false);
            mma_commit(bar);
        }
        if (!wait_mma(bar, phase)) { aborted = true; break; }
        // prefetch the next chunk's v (its buffer is free now)
        if (has_next) {
            load_v(smem, v, b, T, t0n, Ln, HV, hv, tid);
            cp_async_commit();
        }
        {
            float dd[32];
            tmem_ld32(tl + kTmWkT + 32 * ih, dd);  // row i = this lane, columns r
            const int i = 32 * wq + lane;
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8)
                *reinterpret_cast<uint4 *>(smem + kOpWK + mnmajor_off(i, 32 * ih + 8 * q8, kD)) =
                    pack_bf16x8(&dd[8 * q8]);
        }
        // S'^T = (diag(exp(G_m)) S)^T as the A operand (bf16)
#pragma unroll
        for (int u8 = 0; u8 < 8; ++u8) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = S[8 * u8 + e] * sEGm[64 * ih + 8 * u8 + e];
            *reinterpret_cast<uint4 *>(smem + kOpST + kmajor_off(j, 64 * ih + 8 * u8, kD)) =
                pack_bf16x8(x);
        }
        fence_async_smem();
        tc_fence_before_sync();
        __syncthreads();

        // ---------------- MMA batch 3: U^T -= S'^T (T'Lk)^T,  O^T = S'^T Lq^T
        if (tid == 0) {
            tc_fence_after_sync();
            gemm(tmem + kTmUT, sbase + kOpST, 128, kD * 16, sbase + kOpWK, 128, kD * 16,
                 idesc_bf16(128, 64, false, true, true), kD / 16, true);
            gemm(tmem + kTmOT, sbase + kOpST, 128, kD * 16, sbase + kOpL + 16384, 128, kD * 16,
                 idesc_bf16(128, 64, false, false, false), kD / 16, false);
            mma_commit(bar);
        }
        if (!wait_mma(bar, phase)) { aborted = true; break; }
        {
            float dd[32];
            tmem_ld32(tl + kTmUT + 32 * ih, dd);
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8)
                *reinterpret_cast<uint4 *>(smem + kOpUT + kmajor_off(j, 32 * ih + 8 * q8, kC)) =
                    pack_bf16x8(&dd[8 * q8]);
        }
        fence_async_smem();
        tc_fence_before_sync();
        __syncthreads();

        // ---------------- MMA batch 4: O^T += U^T P^T,  dS^T = U^T R (R read MN-major)
        if (tid == 0) {
            tc_fence_after_sync();
            gemm(tmem + kTmOT, sbase + kOpUT, 128, kC * 16, sbase + kOpP, 128, kC * 16,
                 idesc_bf16(128, 64, false, false, false), kC / 16, true);
            gemm(tmem + kTmDS, sbase + kOpUT, 128, kC * 16, sbase + kOpR, kD * 16, 128,
                 idesc_bf16(128, 128, false, true, false), kC / 16, false);
            mma_commit(bar);
        }
        if (!wait_mma(bar, phase)) { aborted = true; break; }
        {
            float dd[32];
            tmem_ld32(tl + kTmDS + 64 * ih, dd);
#pragma unroll
            for (int u = 0; u < 32; ++u) {
                const int i = 64 * ih + u;
                S[u] = fmaf(sGamL[i], S[u], sCL[i] * dd[u]);
            }
            tmem_ld32(tl + kTmDS + 64 * ih + 32, dd);
#pragma unroll
            for (int u = 0; u < 32; ++u) {
                const int i = 64 * ih + 32 + u;
                S[32 + u] = fmaf(sGamL[i], S[32 + u], sCL[i] * dd[u]);
            }
            // O^T -> bf16 O [r][j] staging
            tmem_ld32(tl + kTmOT + 32 * ih, dd);
            __nv_bfloat16 *stg = reinterpret_cast<__nv_bfloat16 *>(smem + kStage);
#pragma unroll
            for (int u = 0; u < 32; ++u) stg[(32 * ih + u) * kD + j] = __float2bfloat16_rn(dd[u]);
        }
        tc_fence_before_sync();
        __syncthreads();
        // coalesced 16-byte stores of the chunk's output rows
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int id = tid + kThreads * it;  // 0..1023
            const int r = id >> 4, cc = id & 15;
            if (r < L)
                *reinterpret_cast<uint4 *>(out + (((size_t)b * T + t0 + r) * HV + hv) * kD + cc * 8) =
                    *reinterpret_cast<const uint4 *>(smem + kStage + r * 256 + cc * 16);
        }
    }

    cp_async_wait0();
    if (aborted) {
        if (tid == 0) atomicOr(dev_error, 1);
    } else if (STORE_HT) {
#pragma unroll
        for (int u = 0; u < 64; ++u) ht[((size_t)head * kD + 64 * ih + u) * kD + j] = S[u];
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

bool tc_prefill_supported(const Problem &p) {
    return p.bf16 && p.dk == kD && p.dv == kD && p.chunk == kC;
}

cudaError_t launch_tc_prefill(const Problem &p, int *dev_error, cudaStream_t stream) {
    const long long blocks = (long long)p.B * p.HV;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(p.q);
    const __nv_bfloat16 *k = static_cast<const __nv_bfloat16 *>(p.k);
    const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(p.v);
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);
    auto run = [&](auto kernel) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        trace_begin(kKernFused, stream);
        kernel<<<(unsigned)blocks, kThreads, kSmemBytes, stream>>>(q, k, v, p.g, p.beta, p.h0, out,
                                                                  p.ht, p.T, p.HK, p.HV, dev_error);
        trace_end(kKernFused, stream);
        return cudaGetLastError();
    };
    if (p.h0 && p.ht) return run(gdr_prefill_tc_kernel<true, true>);
    if (p.h0) return run(gdr_prefill_tc_kernel<true, false>);
    if (p.ht) return run(gdr_prefill_tc_kernel<false, true>);
    return run(gdr_prefill_tc_kernel<false, false>);
}

}  // namespace gdr
