// prefill_tc.cu -- chunkwise WY/UT prefill on the Blackwell tensor cores
// (tcgen05 MMA, TMEM accumulators) for bf16 q/k/v with dk = dv = 128 and
// chunks of 64 tokens, fused into one kernel.
//
// Method: page "Reorder channelwise gated delta rule chunked hot loops for
// autovectorization" (pytorch/executorch PR #21021), second commit summary --
// per chunk: per-channel log-decay prefix sums, the causal query/key terms,
// the beta-folded unit-lower triangular transform, WY pseudo-keys and
// pseudo-values, and the state carried to the next chunk, with a ragged last
// chunk through the same code.  The block forward substitution of the
// triangular transform (16 x 16 diagonal-block inverses, then off-diagonal
// blocks) follows the block-TRSM structure of trymirai/uzu PR #576
// ("Support TreeUpdateSolve kernel", commit summary).
//
// Algebra per chunk of L <= 64 tokens (r, s local token indices; S the state
// at the chunk start; G the inclusive per-channel prefix sum of g):
//   A[r,s] = beta_r sum_i k_ri k_si exp(G_ri - G_si)   (s < r)
//   P[r,s] =        sum_i q_ri k_si exp(G_ri - G_si)   (s <= r)
//   T'     = (I + A)^-1 diag(beta)
//   Wk     = T' (exp(G) * K),   Wv = T' V
//   U      = Wv - Wk S
//   O      = (exp(G) * Q) S + P U
//   S     <- diag(exp(G_L)) S + (exp(G_L - G) * K)^T U
//
// GB300 mapping.  One CTA (8 warps) per (batch, value head) walks that head's
// chunks in order; the float32 state never leaves registers (thread = one
// value column j, 64 of the 128 key rows).  The state-dependent products are
// computed transposed so that M = dv = 128 fills the MMA:
//   U^T = Wv^T - S^T Wk^T,  O^T = S^T Qt^T + U^T P^T,  dS^T = U^T Kh.
// Every operand is bf16 in shared memory in the interleaved (no-swizzle)
// core-matrix layout (sm100_ptx.cuh); every accumulator is float32 in TMEM.
// Per chunk the tensor core runs 7 GEMMs (gram, W_k^T, W_v^T, U^T, two for
// O^T, dS^T); the 64 x 64 triangular inverse runs in float32 on CUDA cores.
//
// The decays exp(G_r - G_s) of the gram are factored around a reference row m
// of the chunk: exp(G_r - G_m) * exp(G_m - G_s).  While every channel decays
// by at most 80 nats between the first token and m and between m and the last
// token, both factors are finite in bf16/f32 and the product is exact to
// rounding.  A chunk outside that range (decay stronger than ~2.5 nats per
// token sustained over 32 tokens) takes an exact pairwise path on CUDA cores
// for A and P instead, so the result is correct for any g <= 0.
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
constexpr uint32_t kRawK = 0;                 // bf16 [64][128] row-major
constexpr uint32_t kRawQ = kRawK + 16384;     // bf16 [64][128] row-major
constexpr uint32_t kOpV = kRawQ + 16384;      // V as MN-major A (k = s, mn = j), K extent 64
constexpr uint32_t kG = kOpV + 16384;         // f32 [64][128]; later T (f32 64x64) and X
constexpr uint32_t kT32 = kG;                 //   f32 [64][64]
constexpr uint32_t kX32 = kG + 16384;         //   f32 [3][16][16] scratch of the block solve
constexpr uint32_t kLR = kG + 32768;          // 48 KB region:
constexpr uint32_t kOpL = kLR;                //   gram A operand [128][128] K-major (K rows | Q rows)
constexpr uint32_t kOpR = kLR + 32768;        //   gram B operand [64][128] K-major
constexpr uint32_t kA32 = kLR;                //   then: f32 A [64][64] (swizzled)
constexpr uint32_t kOpWK = kLR + 16384;       //   then: Wk as MN-major B (k = i, mn = r), K extent 128
constexpr uint32_t kOpUT = kLR + 32768;       //   then: U^T as K-major A [128 j][64 r]
constexpr uint32_t kOpKT = kLR + 49152;       // Kt as MN-major A (k = s, mn = i), K extent 64
constexpr uint32_t kOpQT = kOpKT + 16384;     // Qt as K-major B [64 r][128 i]
constexpr uint32_t kOpKH = kOpQT + 16384;     // Kh as MN-major B (k = r, mn = i), K extent 64
constexpr uint32_t kOpT = kOpKH + 16384;      // T' as K-major B [64 r][64 s]
constexpr uint32_t kOpP = kOpT + 8192;        // P as K-major B [64 r][64 s]
constexpr uint32_t kOpST = kOpP + 8192;       // S^T as K-major A [128 j][128 i]
constexpr uint32_t kSmall = kOpST + 32768;
constexpr uint32_t kBeta = kSmall;            // f32 [64]
constexpr uint32_t kGm = kBeta + 256;         // f32 [128]  G at the reference row
constexpr uint32_t kEGm = kGm + 512;          // f32 [128]  exp(G_m)
constexpr uint32_t kCL = kEGm + 512;          // f32 [128]  exp(G_last - G_m)
constexpr uint32_t kGamL = kCL + 512;         // f32 [128]  exp(G_last)
constexpr uint32_t kTot = kGamL;              // f32 [128]  prefix-sum carry (before kGamL is set)
constexpr uint32_t kBar = kGamL + 512;        // mbarrier (8 B)
constexpr uint32_t kTmemSlot = kBar + 8;      // u32
constexpr uint32_t kSmemBytes = kTmemSlot + 8;
static_assert(kSmemBytes <= 232448, "shared memory budget");

// ---- TMEM columns (float32 accumulators, lane = M row)
constexpr uint32_t kTmGram = 0;     // [128 x 64]: rows 0-63 K-gram, 64-127 Q-gram
constexpr uint32_t kTmWkT = 64;     // [128 i x 64 r]
constexpr uint32_t kTmUT = 128;     // [128 j x 64 r]
constexpr uint32_t kTmOT = 192;     // [128 j x 64 r]
constexpr uint32_t kTmDS = 256;     // [128 j x 128 i]
constexpr uint32_t kTmemCols = 512;

// operand descriptor byte strides
constexpr uint32_t kLBO = 128;
__device__ __forceinline__ uint32_t sbo_for(int k_extent) { return (uint32_t)k_extent * 16u; }

// A (f32 64 x 64) with an XOR swizzle so row-wise and column-wise walks stay conflict-free
__device__ __forceinline__ int a_idx(int r, int s) { return r * 64 + (s ^ (r & 31)); }

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

// Issues the K-steps of one GEMM: D (+)= A * B^T over k_steps * 16 of K.
__device__ __forceinline__ void gemm(uint32_t d_tmem, uint32_t a_addr, uint32_t a_sbo,
                                     uint32_t b_addr, uint32_t b_sbo, uint32_t idesc,
                                     int k_steps, bool accumulate_first) {
    for (int ks = 0; ks < k_steps; ++ks) {
        const uint64_t ad = smem_desc(a_addr + ks * 2 * kLBO, kLBO, a_sbo);
        const uint64_t bd = smem_desc(b_addr + ks * 2 * kLBO, kLBO, b_sbo);
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
    const int ih = warp >> 2;       // which half of the 128 key channels / 64 tokens
    const int head = blockIdx.x;    // b * HV + hv
    const int hv = head % HV, b = head / HV;
    const int hk = hv / (HV / HK);
    const int j = 32 * wq + lane;   // this thread's value column (TMEM lane)

    float *sbeta = reinterpret_cast<float *>(smem + kBeta);
    float *sGm = reinterpret_cast<float *>(smem + kGm);
    float *sEGm = reinterpret_cast<float *>(smem + kEGm);
    float *sCL = reinterpret_cast<float *>(smem + kCL);
    float *sGamL = reinterpret_cast<float *>(smem + kGamL);
    float *sTot = reinterpret_cast<float *>(smem + kTot);
    float *sG = reinterpret_cast<float *>(smem + kG);
    float *sA = reinterpret_cast<float *>(smem + kA32);
    float *sT = reinterpret_cast<float *>(smem + kT32);
    float *sX = reinterpret_cast<float *>(smem + kX32);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kTmemSlot);

    if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
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

    const int NC = (T + kC - 1) / kC;
    for (int c = 0; c < NC; ++c) {
        const int t0 = c * kC;
        const int L = min(kC, T - t0);
        const int m = (L - 1) / 2;  // reference row of the gram factorisation

        // ---------------- load the chunk (16-byte cp.async; zero rows >= L)
        const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int id = tid + kThreads * it;  // 0..1023
            const int r = id >> 4, cc = id & 15;
            unsigned char *dk_ = smem + kRawK + r * 256 + cc * 16;
            unsigned char *dq_ = smem + kRawQ + r * 256 + cc * 16;
            unsigned char *dv_ = smem + kOpV + mnmajor_off(r, cc * 8, kC);
            if (r < L) {
                const size_t tk = ((size_t)b * T + t0 + r) * HK + hk;
                const size_t tv = ((size_t)b * T + t0 + r) * HV + hv;
                cp_async16(dk_, k + tk * kD + cc * 8);
                cp_async16(dq_, q + tk * kD + cc * 8);
                cp_async16(dv_, v + tv * kD + cc * 8);
            } else {
                *reinterpret_cast<uint4 *>(dk_) = zero4;
                *reinterpret_cast<uint4 *>(dq_) = zero4;
                *reinterpret_cast<uint4 *>(dv_) = zero4;
            }
        }
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int id = tid + kThreads * it;  // 0..2047
            const int r = id >> 5, cc = id & 31;
            unsigned char *dg = smem + kG + r * 512 + cc * 16;
            if (r < L)
                cp_async16(dg, g + (((size_t)b * T + t0 + r) * HV + hv) * kD + cc * 4);
            else
                *reinterpret_cast<uint4 *>(dg) = zero4;
        }
        if (tid < kC) sbeta[tid] = tid < L ? beta[((size_t)b * T + t0 + tid) * HV + hv] : 0.f;
        cp_async_wait_all();
        __syncthreads();

        // ---------------- per-channel prefix sums of g (two halves of 32 rows)
        {
            const int i = tid & 127, hh = tid >> 7;
            float x[32];
#pragma unroll
            for (int r = 0; r < 32; ++r) x[r] = sG[(32 * hh + r) * kD + i];
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
            for (int r = 0; r < 32; ++r) sG[(32 * hh + r) * kD + i] = x[r];
        }
        __syncthreads();
        int bad = 0;
        if (tid < kD) {
            const int i = tid;
            const float g0 = sG[i], gm = sG[m * kD + i], gl = sG[(L - 1) * kD + i];
            sGm[i] = gm;
            sEGm[i] = __expf(gm);
            sCL[i] = __expf(gl - gm);
            sGamL[i] = __expf(gl);
            bad = (g0 - gm > kRangeNats) || (gm - gl > kRangeNats);
        }
        const bool slow = __syncthreads_or(bad) != 0;

        // ---------------- operands (bf16, core-matrix layouts)
#pragma unroll 1
        for (int it = 0; it < 4; ++it) {
            const int id = tid + kThreads * it;  // 0..1023
            const int r = ((id >> 7) << 3) | (id & 7);
            const int ch = ((id >> 3) & 15) * 8;
            float kv[8], qv[8], Gv[8];
            unpack_bf16x8(*reinterpret_cast<const uint4 *>(smem + kRawK + r * 256 + ch * 2), kv);
            unpack_bf16x8(*reinterpret_cast<const uint4 *>(smem + kRawQ + r * 256 + ch * 2), qv);
            const float4 g_lo = *reinterpret_cast<const float4 *>(sG + r * kD + ch);
            const float4 g_hi = *reinterpret_cast<const float4 *>(sG + r * kD + ch + 4);
            Gv[0] = g_lo.x; Gv[1] = g_lo.y; Gv[2] = g_lo.z; Gv[3] = g_lo.w;
            Gv[4] = g_hi.x; Gv[5] = g_hi.y; Gv[6] = g_hi.z; Gv[7] = g_hi.w;
            float kt[8], qt[8], kh[8];
            if (!slow) {
                float lk[8], lq[8], rk[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float d = Gv[e] - sGm[ch + e];
                    const float el = __expf(d), er = __expf(-d);
                    lk[e] = kv[e] * el;
                    lq[e] = qv[e] * el;
                    rk[e] = kv[e] * er;
                    kt[e] = lk[e] * sEGm[ch + e];
                    qt[e] = lq[e] * sEGm[ch + e];
                    kh[e] = rk[e] * sCL[ch + e];
                }
                *reinterpret_cast<uint4 *>(smem + kOpL + kmajor_off(r, ch, kD)) = pack_bf16x8(lk);
                *reinterpret_cast<uint4 *>(smem + kOpL + kmajor_off(64 + r, ch, kD)) = pack_bf16x8(lq);
                *reinterpret_cast<uint4 *>(smem + kOpR + kmajor_off(r, ch, kD)) = pack_bf16x8(rk);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float eg = __expf(Gv[e]);
                    kt[e] = kv[e] * eg;
                    qt[e] = qv[e] * eg;
                    kh[e] = kv[e] * __expf(sG[(L - 1) * kD + ch + e] - Gv[e]);
                }
            }
            *reinterpret_cast<uint4 *>(smem + kOpKT + mnmajor_off(r, ch, kC)) = pack_bf16x8(kt);
            *reinterpret_cast<uint4 *>(smem + kOpQT + kmajor_off(r, ch, kD)) = pack_bf16x8(qt);
            *reinterpret_cast<uint4 *>(smem + kOpKH + mnmajor_off(r, ch, kC)) = pack_bf16x8(kh);
        }
        // S^T (bf16) as the A operand of the state products
#pragma unroll
        for (int u8 = 0; u8 < 8; ++u8)
            *reinterpret_cast<uint4 *>(smem + kOpST + kmajor_off(j, 64 * ih + 8 * u8, kD)) =
                pack_bf16x8(&S[8 * u8]);
        fence_async_smem();
        __syncthreads();

        // ---------------- MMA batch 1: gram = [K; Q]-left x K-right^T,  O^T = S^T Qt^T
        if (tid == 0) {
            tc_fence_after_sync();
            if (!slow)
                gemm(tmem + kTmGram, sbase + kOpL, sbo_for(kD), sbase + kOpR, sbo_for(kD),
                     idesc_bf16(128, 64, false, false, false), kD / 16, false);
            gemm(tmem + kTmOT, sbase + kOpST, sbo_for(kD), sbase + kOpQT, sbo_for(kD),
                 idesc_bf16(128, 64, false, false, false), kD / 16, false);
            mma_commit(bar);
        }
        if (!wait_mma(bar, phase)) { aborted = true; break; }

        // ---------------- A (f32, beta-folded, strictly lower) and P (bf16, causal)
        if (!slow) {
            float d[32];
            tmem_ld32(tl + kTmGram + 32 * ih, d);
            const int row = 32 * wq + lane;
            if (row < kC) {
                const int r = row;
                const float br = sbeta[r];
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    const int s = 32 * ih + u;
                    sA[a_idx(r, s)] = (s < r && r < L) ? br * d[u] : 0.f;
                }
            } else {
                const int r = row - kC;
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    const int s = 32 * ih + u;
                    d[u] = (s <= r && r < L) ? d[u] : 0.f;
                }
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8)
                    *reinterpret_cast<uint4 *>(smem + kOpP + kmajor_off(r, 32 * ih + 8 * q8, kC)) =
                        pack_bf16x8(&d[8 * q8]);
            }
        } else {
            // exact pairwise decays on CUDA cores (every exponent <= 0)
            const __nv_bfloat16 *rk = reinterpret_cast<const __nv_bfloat16 *>(smem + kRawK);
            const __nv_bfloat16 *rq = reinterpret_cast<const __nv_bfloat16 *>(smem + kRawQ);
            __nv_bfloat16 *op = reinterpret_cast<__nv_bfloat16 *>(smem + kOpP);
            for (int idx = tid; idx < kC * kC; idx += kThreads) {
                const int r = idx >> 6, s = idx & 63;
                float a = 0.f, p = 0.f;
                if (s <= r && r < L) {
                    for (int i = 0; i < kD; ++i) {
                        const float e = __expf(sG[r * kD + i] - sG[s * kD + i]);
                        const float kse = __bfloat162float(rk[s * kD + i]) * e;
                        a = fmaf(__bfloat162float(rk[r * kD + i]), kse, a);
                        p = fmaf(__bfloat162float(rq[r * kD + i]), kse, p);
                    }
                }
                sA[a_idx(r, s)] = (s < r) ? sbeta[r] * a : 0.f;
                op[kmajor_off(r, s, kC) >> 1] = __float2bfloat16_rn(p);
            }
        }
        tc_fence_before_sync();
        __syncthreads();

        // ---------------- T = (I + A)^-1 by block forward substitution (f32)
        if (tid < 64) {
            // diagonal 16 x 16 blocks: thread (I, jj) solves column jj of block I
            const int I = tid >> 4, jj = tid & 15;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float acc = (r == jj) ? 1.f : 0.f;
#pragma unroll
                for (int s = 0; s < r; ++s) acc = fmaf(-sA[a_idx(16 * I + r, 16 * I + s)], x[s], acc);
                x[r] = acc;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) sT[(16 * I + r) * 64 + 16 * I + jj] = x[r];
        }
        __syncthreads();
#pragma unroll 1
        for (int dlev = 1; dlev < 4; ++dlev) {
            const int nblk = 4 - dlev;
            // X_IJ = sum_{M=J}^{I-1} A_IM T_MJ  for I = J + dlev
            for (int o = tid; o < nblk * 256; o += kThreads) {
                const int J = o >> 8, rr = (o >> 4) & 15, cc = o & 15;
                const int I = J + dlev;
                float acc = 0.f;
                for (int M = J; M < I; ++M) {
#pragma unroll
                    for (int kk = 0; kk < 16; ++kk)
                        acc = fmaf(sA[a_idx(16 * I + rr, 16 * M + kk)],
                                   sT[(16 * M + kk) * 64 + 16 * J + cc], acc);
                }
                sX[o] = acc;
            }
            __syncthreads();
            // T_IJ = -T_II X_IJ
            for (int o = tid; o < nblk * 256; o += kThreads) {
                const int J = o >> 8, rr = (o >> 4) & 15, cc = o & 15;
                const int I = J + dlev;
                float acc = 0.f;
                for (int kk = 0; kk <= rr; ++kk)
                    acc = fmaf(sT[(16 * I + rr) * 64 + 16 * I + kk], sX[(J << 8) + kk * 16 + cc], acc);
                sT[(16 * I + rr) * 64 + 16 * J + cc] = -acc;
            }
            __syncthreads();
        }
        // T' = T diag(beta) as bf16 (zero above the diagonal)
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const int id = tid + kThreads * it;  // 0..511
            const int r = id >> 3, s0 = (id & 7) * 8;
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int s = s0 + e;
                x[e] = (s <= r) ? sT[r * 64 + s] * sbeta[s] : 0.f;
            }
            *reinterpret_cast<uint4 *>(smem + kOpT + kmajor_off(r, s0, kC)) = pack_bf16x8(x);
        }
        fence_async_smem();
        __syncthreads();

        // ---------------- MMA batch 2: Wk^T = Kt^T T'^T,  U^T = V^T T'^T (= Wv^T)
        if (tid == 0) {
            tc_fence_after_sync();
            gemm(tmem + kTmWkT, sbase + kOpKT, sbo_for(kC), sbase + kOpT, sbo_for(kC),
                 idesc_bf16(128, 64, true, false, false), kC / 16, false);
            gemm(tmem + kTmUT, sbase + kOpV, sbo_for(kC), sbase + kOpT, sbo_for(kC),
                 idesc_bf16(128, 64, true, false, false), kC / 16, false);
            mma_commit(bar);
        }
        if (!wait_mma(bar, phase)) { aborted = true; break; }
        {
            float d[32];
            tmem_ld32(tl + kTmWkT + 32 * ih, d);  // row i = j-th lane, columns r
            const int i = 32 * wq + lane;
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8)
                *reinterpret_cast<uint4 *>(smem + kOpWK + mnmajor_off(i, 32 * ih + 8 * q8, kD)) =
                    pack_bf16x8(&d[8 * q8]);
        }
        fence_async_smem();
        tc_fence_before_sync();
        __syncthreads();

        // ---------------- MMA batch 3: U^T -= S^T Wk^T
        if (tid == 0) {
            tc_fence_after_sync();
            gemm(tmem + kTmUT, sbase + kOpST, sbo_for(kD), sbase + kOpWK, sbo_for(kD),
                 idesc_bf16(128, 64, false, true, true), kD / 16, true);
            mma_commit(bar);
        }
        if (!wait_mma(bar, phase)) { aborted = true; break; }
        {
            float d[32];
            tmem_ld32(tl + kTmUT + 32 * ih, d);
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8)
                *reinterpret_cast<uint4 *>(smem + kOpUT + kmajor_off(j, 32 * ih + 8 * q8, kC)) =
                    pack_bf16x8(&d[8 * q8]);
        }
        fence_async_smem();
        tc_fence_before_sync();
        __syncthreads();

        // ---------------- MMA batch 4: O^T += U^T P^T,  dS^T = U^T Kh
        if (tid == 0) {
            tc_fence_after_sync();
            gemm(tmem + kTmOT, sbase + kOpUT, sbo_for(kC), sbase + kOpP, sbo_for(kC),
                 idesc_bf16(128, 64, false, false, false), kC / 16, true);
            gemm(tmem + kTmDS, sbase + kOpUT, sbo_for(kC), sbase + kOpKH, sbo_for(kC),
                 idesc_bf16(128, 128, false, true, false), kC / 16, false);
            mma_commit(bar);
        }
        if (!wait_mma(bar, phase)) { aborted = true; break; }
        {
            float d[32];
            tmem_ld32(tl + kTmDS + 64 * ih, d);
#pragma unroll
            for (int u = 0; u < 32; ++u) S[u] = fmaf(sGamL[64 * ih + u], S[u], d[u]);
            tmem_ld32(tl + kTmDS + 64 * ih + 32, d);
#pragma unroll
            for (int u = 0; u < 32; ++u) S[32 + u] = fmaf(sGamL[64 * ih + 32 + u], S[32 + u], d[u]);
            tmem_ld32(tl + kTmOT + 32 * ih, d);
#pragma unroll
            for (int u = 0; u < 32; ++u) {
                const int r = 32 * ih + u;
                if (r < L)
                    out[(((size_t)b * T + t0 + r) * HV + hv) * kD + j] = __float2bfloat16_rn(d[u]);
            }
        }
        tc_fence_before_sync();
        __syncthreads();
    }

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
