// tree_blocked.cu -- tree verification of up to 512 draft tokens: the whole
// tree as one unit-lower system, solved 16 rows at a time.
//
// Page "Support TreeUpdateSolve kernel" (trymirai/uzu PR #576), commit
// summary: a gram of block pairs, 16 x 16 diagonal blocks, and a block
// forward substitution (a "pure block TRSM") whose right-hand side starts
// from kh0 = the decayed keys against h0; its review thread: the gram per
// key head when the gate is one scalar per token (shared by the key head's
// value heads).  Page "Reorder channelwise gated delta rule chunked hot
// loops" (pytorch/executorch): the chunkwise WY form, here over a tree's
// ancestor relation instead of the causal order.
//
// For one tree and value head, with G_t the sum of the log-decays g over t's
// root path (t included) and anc(t) its strict ancestors:
//   A_rs = beta_r sum_c k_r[c] k_s[c] exp(G_r[c] - G_s[c])        s in anc(r)
//   P_rs =        sum_c q_r[c] k_s[c] exp(G_r[c] - G_s[c])        s in anc(r) or s = r
//   kh0_r = (k_r exp(G_r)) h0,   qh0_r = (q_r exp(G_r)) h0
//   U_r  = beta_r (v_r - kh0_r) - sum_{s in anc(r)} A_rs U_s      (forward substitution)
//   o_r  = qh0_r + sum_{s in anc(r) or s = r} P_rs U_s
// which is the token recurrence run along each root path (tokens precede
// their descendants, so the system is unit lower triangular).
//
// Launches (everything but the substitution runs in parallel over blocks):
//  gdr_tree_mask_kernel   strict-ancestor bitmasks, one CTA per tree shape;
//  gdr_tree_path_kernel   G (log2 units), 8 key channels per CTA;
//    both by pointer jumping (ceil(log2 T) rounds);
//  gdr_tree_gram_kernel   one CTA per (tree, head, 16-row block I): -A_IJ and
//                         P_IJ for every J <= I holding an ancestor pair, as
//                         bf16 mma.sync fragments, A_II in f32, and a flag
//                         per block pair; a scalar gate may run it per key
//                         head, the raw products shared by its value heads;
//  gdr_tree_solve_kernel  one CTA per (tree, value head, dv part) walks the
//                         blocks in order: kh0, qh0 from h0, the right-hand
//                         side from the earlier blocks' U, U_I by forward
//                         substitution through A_II in f32, then o.  Each
//                         block's fragments are copied in (cp.async) while its
//                         h0 products run.
// Decay factors of a block pair are split about a per-channel reference, the
// largest G over the row block's tokens: row operands take exp(G_r - Gref)
// <= 1, column operands exp(Gref - G_s), which for an ancestor s of a row of
// the block is at most the block's spread max_r (Gref - G_r).  A row block
// spread over more than 60 nats runs one pass per row instead, each row its
// own reference (column factors <= 1).  f32 q/k/v carry every tensor-core
// operand as a bf16 pair hi + lo and every product as hi hi + hi lo + lo hi
// (BF16x3); bf16 q/k/v use one bf16 product.
#include <string.h>

#include <algorithm>

#include "common.cuh"

namespace gdr {
namespace {

constexpr int kTreeThreads = 256;
constexpr int kTreeMaxT = 512;
constexpr float kLog2eT = 1.4426950408889634f;
// spread limit of a factored row block, and the clamp of every exponent
// (log2 units): factors stay finite whatever the masked pairs hold
constexpr float kSpreadLog2 = 60.f * kLog2eT;
constexpr float kClampLog2 = 100.f;
constexpr int kPathCh = 8;  // key channels per path-sum CTA

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint32_t bf2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
// x = hi + lo in bf16 pairs (lo = the rounding error of hi, rounded)
template <bool SPLIT>
__device__ __forceinline__ void pack2(float a, float b, uint32_t &hi, uint32_t &lo) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    hi = *reinterpret_cast<uint32_t *>(&h);
    if (SPLIT) {
        const float2 f = __bfloat1622float2(h);
        lo = bf2(a - f.x, b - f.y);
    } else {
        lo = 0u;
    }
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <bool SPLIT>
__device__ __forceinline__ void mma3(float (&c)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4],
                                     uint32_t bh0, uint32_t bh1, uint32_t bl0, uint32_t bl1) {
    mma16816(c, ah, bh0, bh1);
    if (SPLIT) {
        mma16816(c, ah, bl0, bl1);
        mma16816(c, al, bh0, bh1);
    }
}

__device__ __forceinline__ float2 unpack2(uint32_t w) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w));
}
// Two consecutive q/k/v elements as f32.
__device__ __forceinline__ float2 ld2(const float *p) { return *reinterpret_cast<const float2 *>(p); }
__device__ __forceinline__ float2 ld2(const __nv_bfloat16 *p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
}
__device__ __forceinline__ void st2(float *p, float a, float b) {
    *reinterpret_cast<float2 *>(p) = make_float2(a, b);
}
__device__ __forceinline__ void st2(__nv_bfloat16 *p, float a, float b) {
    *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(a, b);
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__host__ __device__ inline int tri(int I, int J) { return I * (I + 1) / 2 + J; }

// ------------------------------------------------------------------ masks
// grid B, one thread per (padded) token: the strict-ancestor bitmasks of
// batch element b, [Tp][Tp / 32], by pointer jumping with the masks in
// registers.
__global__ void __launch_bounds__(kTreeMaxT)
    gdr_tree_mask_kernel(const int *__restrict__ parent, uint32_t *__restrict__ anc, int T, int Tp,
                         int rounds) {
    __shared__ int sP[kTreeMaxT];
    __shared__ uint32_t sM[kTreeMaxT * (kTreeMaxT / 32)];
    const int b = blockIdx.x, t = threadIdx.x, NW = Tp / 32;
    int p = t < T ? parent[(size_t)b * T + t] : -1;
    uint32_t m[kTreeMaxT / 32];
#pragma unroll
    for (int w = 0; w < kTreeMaxT / 32; ++w) m[w] = (p >= 0 && (p >> 5) == w) ? (1u << (p & 31)) : 0u;
    for (int r = 0; r < rounds; ++r) {
        sP[t] = p;
#pragma unroll
        for (int w = 0; w < kTreeMaxT / 32; ++w)
            if (w < NW) sM[w * Tp + t] = m[w];
        __syncthreads();
        if (p >= 0) {
#pragma unroll
            for (int w = 0; w < kTreeMaxT / 32; ++w)
                if (w < NW) m[w] |= sM[w * Tp + p];
            p = sP[p];
        }
        __syncthreads();
    }
#pragma unroll
    for (int w = 0; w < kTreeMaxT / 32; ++w)
        if (w < NW) anc[((size_t)b * Tp + t) * NW + w] = m[w];
}

// ------------------------------------------------------------------ path sums
// grid (dkG / CH, B * HV), one thread per (padded) token: channels
// [CH x, CH x + CH) of G for tree (b, hv) by pointer jumping with the sums in
// registers.  Channelwise gates (CH = kPathCh) also leave, per 16-token
// block J, its reference Gref(J) (the largest G of the block's tokens), a
// flag per channel group when the block spreads past the factored limit,
// and the column operands Kh_s = k_s exp(Gref(J) - G_s) (bf16 channel pairs,
// hi then lo for f32 q/k/v).
template <typename IO, int CH, bool SPLIT>
__global__ void __launch_bounds__(kTreeMaxT)
    gdr_tree_path_kernel(const int *__restrict__ parent, const float *__restrict__ g,
                         const IO *__restrict__ k, float *__restrict__ Gp, float *__restrict__ Gref,
                         int *__restrict__ spread, uint32_t *__restrict__ Kh, int T, int Tp, int NBT,
                         int HK, int HV, int dkG, int rounds) {
    __shared__ int sP[kTreeMaxT];
    __shared__ float sG[kTreeMaxT * CH];
    const int tree = blockIdx.y, b = tree / HV, hv = tree % HV, t = threadIdx.x;
    const int c0 = CH * blockIdx.x;
    int p = t < T ? parent[(size_t)b * T + t] : -1;
    float x[CH];
    const float *gr = g + ((size_t)b * T + t) * HV * dkG + (size_t)hv * dkG + c0;
    float *gw = Gp + ((size_t)tree * Tp + t) * dkG + c0;
    if (CH % 4 == 0) {
#pragma unroll
        for (int c = 0; c < CH; c += 4) {
            const float4 v = t < T ? *reinterpret_cast<const float4 *>(gr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            x[c] = v.x * kLog2eT; x[c + 1] = v.y * kLog2eT; x[c + 2] = v.z * kLog2eT; x[c + 3] = v.w * kLog2eT;
        }
    } else {
#pragma unroll
        for (int c = 0; c < CH; ++c) x[c] = t < T ? gr[c] * kLog2eT : 0.f;
    }
    for (int r = 0; r < rounds; ++r) {
        sP[t] = p;
#pragma unroll
        for (int c = 0; c < CH; ++c) sG[c * Tp + t] = x[c];
        __syncthreads();
        if (p >= 0) {
#pragma unroll
            for (int c = 0; c < CH; ++c) x[c] += sG[c * Tp + p];
            p = sP[p];
        }
        __syncthreads();
    }
    if (CH % 4 == 0) {
#pragma unroll
        for (int c = 0; c < CH; c += 4) *reinterpret_cast<float4 *>(gw + c) = make_float4(x[c], x[c + 1], x[c + 2], x[c + 3]);
    } else {
#pragma unroll
        for (int c = 0; c < CH; ++c) gw[c] = x[c];
    }
    if (CH == 1) return;
    // block references: the 16 tokens of a block are one half-warp
    const int J = t >> 4, dk = dkG, ngroups = dkG / CH;
    float ref[CH];
    int bad = 0;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        float mx = t < T ? x[c] : -3.0e38f, mn = t < T ? x[c] : 3.0e38f;
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) {
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        }
        ref[c] = mx;
        bad |= !(mx - mn <= kSpreadLog2);
    }
    if ((t & 15) == 0 && J < NBT) {
#pragma unroll
        for (int c = 0; c < CH; ++c) Gref[((size_t)tree * NBT + J) * dk + c0 + c] = ref[c];
        spread[((size_t)tree * NBT + J) * ngroups + blockIdx.x] = bad;
    }
    // Kh_t over this group's channels
    const IO *kr = k + ((size_t)b * T + t) * HK * dk + (size_t)(hv / (HV / HK)) * dk + c0;
    uint32_t *kh = Kh + ((size_t)tree * Tp + t) * (SPLIT ? dk : dk / 2) + c0 / 2;
    uint32_t whi[CH / 2 > 0 ? CH / 2 : 1], wlo[CH / 2 > 0 ? CH / 2 : 1];
#pragma unroll
    for (int c = 0; c < CH; c += 2) {
        float2 kk = make_float2(0.f, 0.f);
        if (t < T) {
            kk = ld2(kr + c);
            kk.x *= ex2(fminf(ref[c] - x[c], kClampLog2));
            kk.y *= ex2(fminf(ref[c + 1] - x[c + 1], kClampLog2));
        }
        pack2<SPLIT>(kk.x, kk.y, whi[c / 2], wlo[c / 2]);
    }
#pragma unroll
    for (int w = 0; w < CH / 2; w += 4) {
        *reinterpret_cast<uint4 *>(kh + w) = make_uint4(whi[w], whi[w + 1], whi[w + 2], whi[w + 3]);
        if (SPLIT)
            *reinterpret_cast<uint4 *>(kh + dk / 2 + w) = make_uint4(wlo[w], wlo[w + 1], wlo[w + 2], wlo[w + 3]);
    }
}

// ------------------------------------------------------------------ grams
struct GramArgs {
    const void *q, *k;
    const float *beta;
    const float *Gp;      // [B * HV][Tp][dk or 1] path sums, log2 units
    const float *Gref;    // [B * HV][NBT][dk] block references (channelwise)
    const int *spread;    // [B * HV][NBT][dk / kPathCh] block spread flags
    const uint32_t *Kh;   // [B * HV][Tp][dk / 2 (x2 split)] column operands
    const uint32_t *anc;  // [B][Tp][Tp / 32]
    uint32_t *frags;      // [B * HV][NTRI][2 (-A, P)][m (hi, lo)][4][32]
    int *nz;              // [B * HV][NTRI]: the block pair holds an ancestor pair
    float *Ad;            // [B * HV][NBT][16][16] f32 A_II
    int T, Tp, NBT, HK, HV;
};
__host__ __device__ inline int gram_smem_words(int Tp, int dk, bool split, int heads) {
    const int m = split ? 2 : 1, tstride = dk / 2 + 4;
    return 2 * m * 16 * tstride + dk + 16 * (Tp / 32) + 2 * 16 * heads + (kTreeThreads / 32) * dk;
}

// grid (NBT, B * HV), or (NBT, B * HK) with PER_KH (scalar gate: the raw
// products once per key head, then each of its value heads' epilogue).
template <typename IO, int DK, bool SPLIT, bool SCALAR_G, bool PER_KH>
__global__ void __launch_bounds__(kTreeThreads) gdr_tree_gram_kernel(const GramArgs a) {
    extern __shared__ __align__(16) uint32_t sw[];
    constexpr int M = SPLIT ? 2 : 1;
    constexpr int TS = DK / 2 + 4;  // row tile stride (words)
    constexpr int DKG = SCALAR_G ? 1 : DK;
    constexpr int KW = SPLIT ? DK : DK / 2;  // words of one Kh row
    constexpr int NG = DK / kPathCh;
    constexpr int KC = DK / 16 < 4 ? DK / 16 : 4;  // k-steps per batch of loads
    const int T = a.T, Tp = a.Tp, NW = Tp / 32, HV = a.HV, HK = a.HK, Gh = HV / HK;
    const int I = a.NBT - 1 - (int)blockIdx.x;  // the longest rows first
    const int r0 = 16 * I, nrow = min(16, T - r0);
    int b, hk, hv0, nheads;
    if (PER_KH) {
        b = blockIdx.y / HK; hk = blockIdx.y % HK; hv0 = hk * Gh; nheads = Gh;
    } else {
        b = blockIdx.y / HV; hv0 = blockIdx.y % HV; hk = hv0 / Gh; nheads = 1;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3;
    const IO *q = static_cast<const IO *>(a.q);
    const IO *k = static_cast<const IO *>(a.k);
    auto krow = [&](int t) { return k + ((size_t)b * T + t) * HK * DK + (size_t)hk * DK; };
    auto qrow = [&](int t) { return q + ((size_t)b * T + t) * HK * DK + (size_t)hk * DK; };
    const size_t tree0 = (size_t)(b * HV + hv0);
    const float *Gt = a.Gp + tree0 * Tp * DKG;  // first head's G
    uint32_t *sLk = sw;
    uint32_t *sLq = sw + M * 16 * TS;
    float *sGref = reinterpret_cast<float *>(sw + 2 * M * 16 * TS);
    uint32_t *sMask = sw + 2 * M * 16 * TS + DK;
    float *sBeta = reinterpret_cast<float *>(sMask + 16 * NW);  // [heads][16]
    float *sGrow = sBeta + 16 * nheads;                         // [heads][16] scalar gate
    float *sD = sGrow + 16 * nheads + warp * DK;                // this warp's column scale
    const int NTRI = a.NBT * (a.NBT + 1) / 2;

    for (int idx = tid; idx < 16 * nheads; idx += kTreeThreads) {
        const int hh = idx >> 4, r = idx & 15, hv = hv0 + hh;
        const bool in = r < nrow;
        sBeta[idx] = in ? a.beta[((size_t)b * T + r0 + r) * HV + hv] : 0.f;
        if (SCALAR_G) sGrow[idx] = in ? a.Gp[(size_t)(b * HV + hv) * Tp + r0 + r] : 0.f;
    }
    for (int idx = tid; idx < 16 * NW; idx += kTreeThreads) {
        const int r = idx / NW;
        sMask[idx] = r < nrow ? a.anc[((size_t)b * Tp + r0) * NW + idx] : 0u;
    }
    int bad = 0;
    if (!SCALAR_G) {
        for (int c = tid; c < DK; c += kTreeThreads) sGref[c] = a.Gref[(tree0 * a.NBT + I) * DK + c];
        if (tid < NG) bad = a.spread[(tree0 * a.NBT + I) * NG + tid];
    }
    const bool fallback = __syncthreads_or(bad) != 0;
    for (int idx = tid; idx < 16 * (DK / 2); idx += kTreeThreads) {
        const int r = idx / (DK / 2), cp = idx - r * (DK / 2), c = 2 * cp;
        float2 kk = make_float2(0.f, 0.f), qq = kk, e = make_float2(1.f, 1.f);
        if (r < nrow) {
            kk = ld2(krow(r0 + r) + c);
            qq = ld2(qrow(r0 + r) + c);
            if (!SCALAR_G) {
                const float2 gg = *reinterpret_cast<const float2 *>(Gt + (size_t)(r0 + r) * DK + c);
                e = make_float2(ex2(gg.x - sGref[c]), ex2(gg.y - sGref[c + 1]));
            }
        }
        uint32_t hi, lo;
        const int o = r * TS + cp;
        pack2<SPLIT>(kk.x * e.x, kk.y * e.y, hi, lo);
        sLk[o] = hi;
        if (SPLIT) sLk[16 * TS + o] = lo;
        pack2<SPLIT>(qq.x * e.x, qq.y * e.y, hi, lo);
        sLq[o] = hi;
        if (SPLIT) sLq[16 * TS + o] = lo;
    }
    __syncthreads();
#pragma unroll 1
    for (int J = warp; J <= I; J += kTreeThreads / 32) {
        const int sh = 16 * (J & 1);
        const uint32_t f0 = (sMask[gq * NW + (J >> 1)] >> sh) & 0xffffu;
        const uint32_t f1 = (sMask[(gq + 8) * NW + (J >> 1)] >> sh) & 0xffffu;
        const bool any = __any_sync(0xffffffffu, (f0 | f1) != 0u) || J == I;
        if (lane == 0)
            for (int hh = 0; hh < nheads; ++hh) a.nz[(size_t)(tree0 + hh) * NTRI + tri(I, J)] = any;
        if (!any) continue;
        float ca[2][4], cp[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) ca[nt][e] = cp[nt][e] = 0.f;
        // column block J spread past the factored limit: no Kh for it
        bool fj = false;
        if (!SCALAR_G) fj = __any_sync(0xffffffffu, lane < NG && a.spread[(tree0 * a.NBT + J) * NG + lane] != 0);
        if (!SCALAR_G && !fallback && !fj) {
            // exp(Gref(I) - G_s) = exp(Gref(I) - Gref(J)) Kh_s: one factor per channel
            const float *grj = a.Gref + (tree0 * a.NBT + J) * DK;
            for (int c = lane; c < DK; c += 32) sD[c] = ex2(fminf(sGref[c] - grj[c], kClampLog2));
            __syncwarp();
            const uint32_t *khp = a.Kh + (tree0 * Tp + 16 * J) * KW;
#pragma unroll 1
            for (int kb = 0; kb < DK / 16; kb += KC) {
                uint32_t wh[KC][2][2], wl[KC][2][2];
#pragma unroll
                for (int u = 0; u < KC; ++u)
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int o = (8 * nt + gq) * KW + 8 * (kb + u) + tq + 4 * hh;
                            wh[u][nt][hh] = khp[o];
                            wl[u][nt][hh] = SPLIT ? khp[o + DK / 2] : 0u;
                        }
#pragma unroll
                for (int u = 0; u < KC; ++u) {
                    const int ks = kb + u, c0 = 16 * ks + 2 * tq;
                    uint32_t akh[4], akl[4], aqh[4], aql[4];
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        const int o = (gq + 8 * (x & 1)) * TS + 8 * ks + tq + 4 * (x >> 1);
                        akh[x] = sLk[o];
                        aqh[x] = sLq[o];
                        akl[x] = SPLIT ? sLk[16 * TS + o] : 0u;
                        aql[x] = SPLIT ? sLq[16 * TS + o] : 0u;
                    }
                    const float2 d0 = *reinterpret_cast<const float2 *>(sD + c0);
                    const float2 d1 = *reinterpret_cast<const float2 *>(sD + c0 + 8);
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        uint32_t bh[2], bl[2];
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const float2 d = hh ? d1 : d0;
                            float2 f = unpack2(wh[u][nt][hh]);
                            if (SPLIT) {
                                const float2 l = unpack2(wl[u][nt][hh]);
                                f.x += l.x;
                                f.y += l.y;
                            }
                            pack2<SPLIT>(f.x * d.x, f.y * d.y, bh[hh], bl[hh]);
                        }
                        mma3<SPLIT>(ca[nt], akh, akl, bh[0], bh[1], bl[0], bl[1]);
                        mma3<SPLIT>(cp[nt], aqh, aql, bh[0], bh[1], bl[0], bl[1]);
                    }
                }
            }
            __syncwarp();  // sD is rewritten for this warp's next pair
        } else {
            const int npass = (fallback && !SCALAR_G) ? nrow : 1;
#pragma unroll 1
            for (int rho = 0; rho < npass; ++rho) {
#pragma unroll 2
                for (int ks = 0; ks < DK / 16; ++ks) {
                    const int c0 = 16 * ks + 2 * tq;
                    uint32_t akh[4], akl[4], aqh[4], aql[4];
                    float2 gref[2];
                    if (npass == 1) {
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            const int o = (gq + 8 * (x & 1)) * TS + 8 * ks + tq + 4 * (x >> 1);
                            akh[x] = sLk[o];
                            aqh[x] = sLq[o];
                            akl[x] = SPLIT ? sLk[16 * TS + o] : 0u;
                            aql[x] = SPLIT ? sLq[16 * TS + o] : 0u;
                        }
                        if (!SCALAR_G) {
                            gref[0] = *reinterpret_cast<const float2 *>(sGref + c0);
                            gref[1] = *reinterpret_cast<const float2 *>(sGref + c0 + 8);
                        }
                    } else {
                        // one row, its own reference: raw k and q in row rho only
                        const int rr = r0 + rho;
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            const int row = gq + 8 * (x & 1), c = c0 + 8 * (x >> 1);
                            float2 kk = make_float2(0.f, 0.f), qq = kk;
                            if (row == rho) {
                                kk = ld2(krow(rr) + c);
                                qq = ld2(qrow(rr) + c);
                            }
                            pack2<SPLIT>(kk.x, kk.y, akh[x], akl[x]);
                            pack2<SPLIT>(qq.x, qq.y, aqh[x], aql[x]);
                        }
                        gref[0] = *reinterpret_cast<const float2 *>(Gt + (size_t)rr * DK + c0);
                        gref[1] = *reinterpret_cast<const float2 *>(Gt + (size_t)rr * DK + c0 + 8);
                    }
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const int s = 16 * J + 8 * nt + gq;
                        uint32_t bh[2], bl[2];
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int c = c0 + 8 * hh;
                            float2 kk = make_float2(0.f, 0.f);
                            if (s < T) {
                                kk = ld2(krow(s) + c);
                                if (!SCALAR_G) {
                                    const float2 gs = *reinterpret_cast<const float2 *>(Gt + (size_t)s * DK + c);
                                    kk.x *= ex2(fminf(gref[hh].x - gs.x, kClampLog2));
                                    kk.y *= ex2(fminf(gref[hh].y - gs.y, kClampLog2));
                                }
                            }
                            pack2<SPLIT>(kk.x, kk.y, bh[hh], bl[hh]);
                        }
                        mma3<SPLIT>(ca[nt], akh, akl, bh[0], bh[1], bl[0], bl[1]);
                        mma3<SPLIT>(cp[nt], aqh, aql, bh[0], bh[1], bl[0], bl[1]);
                    }
                }
            }
        }
        // epilogue per value head: ancestor mask, beta, scalar decays
#pragma unroll 1
        for (int hh = 0; hh < nheads; ++hh) {
            const size_t tr = tree0 + hh;
            uint32_t *fr = a.frags + (tr * NTRI + tri(I, J)) * (2 * M * 128);
            const float *Gs = a.Gp + tr * Tp;  // scalar gate: this head's G
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int r = gq + 8 * i;
                    const uint32_t f = i ? f1 : f0;
                    float va[2], vp[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int sl = 8 * nt + 2 * tq + e;
                        const bool an = (f >> sl) & 1u;
                        const bool self = J == I && sl == r && r < nrow;
                        float x = ca[nt][2 * i + e], y = cp[nt][2 * i + e];
                        if (SCALAR_G && (an || self)) {
                            const float d = ex2(fminf(sGrow[16 * hh + r] - Gs[16 * J + sl], 0.f));
                            x *= d;
                            y *= d;
                        }
                        va[e] = an ? sBeta[16 * hh + r] * x : 0.f;
                        vp[e] = (an || self) ? y : 0.f;
                        if (J == I) a.Ad[(tr * a.NBT + I) * 256 + r * 16 + sl] = va[e];
                    }
                    const int reg = 2 * nt + i;
                    uint32_t hi, lo;
                    pack2<SPLIT>(-va[0], -va[1], hi, lo);
                    fr[reg * 32 + lane] = hi;
                    if (SPLIT) fr[128 + reg * 32 + lane] = lo;
                    pack2<SPLIT>(vp[0], vp[1], hi, lo);
                    fr[M * 128 + reg * 32 + lane] = hi;
                    if (SPLIT) fr[M * 128 + 128 + reg * 32 + lane] = lo;
                }
            }
        }
    }
}

// ------------------------------------------------------------------ solve
struct SolveArgs {
    const void *q, *k, *v;
    const float *beta, *h0;
    void *out;
    const float *Gp;
    const uint32_t *frags;
    const int *nz;
    const float *Ad;
    int T, Tp, NBT, HK, HV, dv, dvp;
    int nstage;  // 2: the next block's fragments copy in during this one
};
// Shared-memory map (32-bit words); "hi" arrays are followed by their "lo"
// halves when SPLIT.
struct SolveSmem {
    int u, ustride;    // U history: [Tp / 2][ustride] bf16 row pairs
    int h0, hstride;   // h0 part: [dk / 2][hstride] bf16 channel pairs
    int lk0, lq0, tstride;  // row tiles k exp(G), q exp(G): [16][tstride]
    int r, rstride;    // f32 right-hand side [16][rstride]
    int stage, sstride;  // [nstage] x {A_II f32 [256], fragments [NBT][2][m][128]}
    int nz;            // [NTRI] block-pair flags
    int beta;          // [16]
    int words;
};
__host__ __device__ inline SolveSmem solve_smem(int Tp, int NBT, int dk, int dvp, bool split, bool h0,
                                                int nstage) {
    SolveSmem s;
    const int m = split ? 2 : 1;
    int o = 0;
    s.ustride = dvp + 8;
    s.u = o; o += m * (Tp / 2) * s.ustride;
    s.hstride = dvp + 8;
    s.h0 = o; o += h0 ? m * (dk / 2) * s.hstride : 0;
    s.tstride = dk / 2 + 4;
    s.lk0 = o; o += h0 ? m * 16 * s.tstride : 0;
    s.lq0 = o; o += h0 ? m * 16 * s.tstride : 0;
    s.rstride = dvp + 4;
    s.r = o; o += 16 * s.rstride;
    o = (o + 3) & ~3;  // 16-byte aligned for the copies
    s.sstride = 256 + NBT * 2 * m * 128;
    s.stage = o; o += nstage * s.sstride;
    s.nz = o; o += NBT * (NBT + 1) / 2;
    s.beta = o; o += 16;
    s.words = o;
    return s;
}

// One row block's inputs held in registers while the block before it runs.
template <typename IO, int DK>
struct RowPrefetch {
    static constexpr int N = 16 * (DK / 2) / kTreeThreads > 0 ? 16 * (DK / 2) / kTreeThreads : 1;
    float2 k[N], q[N], g[N];
    float2 v[2][2];
    float beta;
};

template <typename IO, int DK, bool SPLIT, bool SCALAR_G>
__global__ void __launch_bounds__(kTreeThreads, 1) gdr_tree_solve_kernel(const SolveArgs a) {
    extern __shared__ __align__(16) uint32_t sw[];
    constexpr int M = SPLIT ? 2 : 1;
    constexpr int DKG = SCALAR_G ? 1 : DK;
    constexpr int FW = 2 * M * 128;  // words of one block pair's fragments
    using RP = RowPrefetch<IO, DK>;
    const int Tp = a.Tp, T = a.T, NBT = a.NBT, NTRI = NBT * (NBT + 1) / 2;
    const bool has_h0 = a.h0 != nullptr;
    const int nstage = a.nstage;
    const SolveSmem L = solve_smem(Tp, NBT, DK, a.dvp, SPLIT, has_h0, nstage);
    const int tree = blockIdx.y, HV = a.HV, b = tree / HV, hv = tree % HV;
    const int hk = hv / (HV / a.HK);
    const int j0 = blockIdx.x * a.dvp, dvp = a.dvp, dv = a.dv;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3;
    const IO *q = static_cast<const IO *>(a.q);
    const IO *k = static_cast<const IO *>(a.k);
    const IO *v = static_cast<const IO *>(a.v);
    IO *out = static_cast<IO *>(a.out);
    const float *Gt = a.Gp + (size_t)tree * Tp * DKG;
    const uint32_t *frg = a.frags + (size_t)tree * NTRI * FW;
    const int lo_u = (Tp / 2) * L.ustride, lo_h = (DK / 2) * L.hstride, lo_t = 16 * L.tstride;
    float *sR = reinterpret_cast<float *>(sw + L.r);
    float *sBeta = reinterpret_cast<float *>(sw + L.beta);
    int *sNz = reinterpret_cast<int *>(sw + L.nz);
    const int n_nt = dvp / 8;  // n-tiles of this part; warp w owns w and w + 8
    auto krow = [&](int t) { return k + ((size_t)b * T + t) * a.HK * DK + (size_t)hk * DK; };
    auto qrow = [&](int t) { return q + ((size_t)b * T + t) * a.HK * DK + (size_t)hk * DK; };

    // the row inputs of block I into registers (zeros past the tree)
    auto prefetch_rows = [&](int I, RP &rp) {
        const int r0 = 16 * I, nrow = min(16, T - r0);
#pragma unroll
        for (int m = 0; m < RP::N; ++m) {
            const int idx = tid + kTreeThreads * m, r = idx / (DK / 2), c = 2 * (idx - r * (DK / 2));
            rp.k[m] = rp.q[m] = rp.g[m] = make_float2(0.f, 0.f);
            if (has_h0 && r < nrow && idx < 16 * (DK / 2)) {
                rp.k[m] = ld2(krow(r0 + r) + c);
                rp.q[m] = ld2(qrow(r0 + r) + c);
                if (SCALAR_G) {
                    const float x = Gt[r0 + r];
                    rp.g[m] = make_float2(x, x);
                } else {
                    rp.g[m] = *reinterpret_cast<const float2 *>(Gt + (size_t)(r0 + r) * DK + c);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int nt = warp + 8 * u, r = gq + 8 * i;
                rp.v[u][i] = make_float2(0.f, 0.f);
                if (nt < n_nt && r < nrow)
                    rp.v[u][i] = ld2(v + ((size_t)b * T + r0 + r) * HV * dv + (size_t)hv * dv + j0 + 8 * nt + 2 * tq);
            }
        rp.beta = tid < nrow ? a.beta[((size_t)b * T + r0 + tid) * HV + hv] : 0.f;
    };
    // block I's fragments (block pairs holding an ancestor pair) and A_II into stage I % nstage
    auto stage_block = [&](int I) {
        uint32_t *st = sw + L.stage + (nstage == 2 ? (I & 1) : 0) * L.sstride;
        if (tid < 64) cp_async16(st + 4 * tid, a.Ad + ((size_t)tree * NBT + I) * 256 + 4 * tid);
        for (int idx = tid; idx < (I + 1) * (FW / 4); idx += kTreeThreads) {
            const int J = idx / (FW / 4), c = idx - J * (FW / 4);
            if (sNz[tri(I, J)]) cp_async16(st + 256 + J * FW + 4 * c, frg + (size_t)tri(I, J) * FW + 4 * c);
        }
        cp_async_commit();
    };

    for (int idx = tid; idx < NTRI; idx += kTreeThreads) sNz[idx] = a.nz[(size_t)tree * NTRI + idx];
    if (has_h0) {
        const float *h = a.h0 + (size_t)tree * DK * dv;
        for (int idx = tid; idx < (DK / 2) * dvp; idx += kTreeThreads) {
            const int cp = idx / dvp, j = idx - cp * dvp;
            uint32_t hi, lo;
            pack2<SPLIT>(h[(size_t)(2 * cp) * dv + j0 + j], h[(size_t)(2 * cp + 1) * dv + j0 + j], hi, lo);
            sw[L.h0 + cp * L.hstride + j] = hi;
            if (SPLIT) sw[L.h0 + lo_h + cp * L.hstride + j] = lo;
        }
    }
    RP cur;
    prefetch_rows(0, cur);
    __syncthreads();  // the block-pair flags are in
    stage_block(0);

#pragma unroll 1
    for (int I = 0; I < NBT; ++I) {
        const int r0 = 16 * I, nrow = min(16, T - r0);
        // ---------------- this block's rows: beta and the h0 tiles k exp(G), q exp(G)
        if (tid < 16) sBeta[tid] = cur.beta;
        if (has_h0) {
#pragma unroll
            for (int m = 0; m < RP::N; ++m) {
                const int idx = tid + kTreeThreads * m, r = idx / (DK / 2), cp = idx - r * (DK / 2);
                if (idx < 16 * (DK / 2)) {
                    const float ex = ex2(cur.g[m].x), ey = ex2(cur.g[m].y);
                    uint32_t hi, lo;
                    const int o = r * L.tstride + cp;
                    pack2<SPLIT>(cur.k[m].x * ex, cur.k[m].y * ey, hi, lo);
                    sw[L.lk0 + o] = hi;
                    if (SPLIT) sw[L.lk0 + lo_t + o] = lo;
                    pack2<SPLIT>(cur.q[m].x * ex, cur.q[m].y * ey, hi, lo);
                    sw[L.lq0 + o] = hi;
                    if (SPLIT) sw[L.lq0 + lo_t + o] = lo;
                }
            }
        }
        float2 vv[2][2];
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int i = 0; i < 2; ++i) vv[u][i] = cur.v[u][i];
        // the next block's rows and fragments start their way in
        if (I + 1 < NBT) {
            prefetch_rows(I + 1, cur);
            if (nstage == 2) stage_block(I + 1);
        }
        __syncthreads();
        // ---------------- kh0, qh0; rhs = beta (v - kh0), o = qh0
        float cr[2][4], co[2][4];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int nt = warp + 8 * u;
            if (nt >= n_nt) break;
#pragma unroll
            for (int e = 0; e < 4; ++e) cr[u][e] = co[u][e] = 0.f;
            const int col = 8 * nt + gq;
            if (has_h0) {
#pragma unroll 4
                for (int ks = 0; ks < DK / 16; ++ks) {
                    uint32_t akh[4], akl[4], aqh[4], aql[4];
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        const int o = (gq + 8 * (x & 1)) * L.tstride + 8 * ks + tq + 4 * (x >> 1);
                        akh[x] = sw[L.lk0 + o];
                        aqh[x] = sw[L.lq0 + o];
                        akl[x] = SPLIT ? sw[L.lk0 + lo_t + o] : 0u;
                        aql[x] = SPLIT ? sw[L.lq0 + lo_t + o] : 0u;
                    }
                    const int o0 = (8 * ks + tq) * L.hstride + col, o1 = o0 + 4 * L.hstride;
                    const uint32_t bh0 = sw[L.h0 + o0], bh1 = sw[L.h0 + o1];
                    const uint32_t bl0 = SPLIT ? sw[L.h0 + lo_h + o0] : 0u;
                    const uint32_t bl1 = SPLIT ? sw[L.h0 + lo_h + o1] : 0u;
                    mma3<SPLIT>(cr[u], akh, akl, bh0, bh1, bl0, bl1);
                    mma3<SPLIT>(co[u], aqh, aql, bh0, bh1, bl0, bl1);
                }
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float br = sBeta[gq + 8 * i];
                cr[u][2 * i] = br * (vv[u][i].x - cr[u][2 * i]);
                cr[u][2 * i + 1] = br * (vv[u][i].y - cr[u][2 * i + 1]);
            }
        }
        // this block's copies are in (the next block's may still be on the way)
        if (nstage == 2 && I + 1 < NBT)
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        else
            cp_async_wait();
        __syncthreads();
        const uint32_t *stg = sw + L.stage + (nstage == 2 ? (I & 1) : 0) * L.sstride;
        const float *sAd = reinterpret_cast<const float *>(stg);
        const uint32_t *sFr = stg + 256;
        // ---------------- the earlier blocks: rhs -= A_IJ U_J, o += P_IJ U_J
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int nt = warp + 8 * u;
            if (nt >= n_nt) break;
            const int col = 8 * nt + gq;
#pragma unroll 2
            for (int J = 0; J < I; ++J) {
                if (!sNz[tri(I, J)]) continue;
                const uint32_t *f = sFr + J * FW;
                uint32_t aah[4], aal[4], pph[4], ppl[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    aah[x] = f[x * 32 + lane];
                    aal[x] = SPLIT ? f[128 + x * 32 + lane] : 0u;
                    pph[x] = f[M * 128 + x * 32 + lane];
                    ppl[x] = SPLIT ? f[M * 128 + 128 + x * 32 + lane] : 0u;
                }
                const int o0 = (8 * J + tq) * L.ustride + col, o1 = o0 + 4 * L.ustride;
                const uint32_t bh0 = sw[L.u + o0], bh1 = sw[L.u + o1];
                const uint32_t bl0 = SPLIT ? sw[L.u + lo_u + o0] : 0u;
                const uint32_t bl1 = SPLIT ? sw[L.u + lo_u + o1] : 0u;
                mma3<SPLIT>(cr[u], aah, aal, bh0, bh1, bl0, bl1);
                mma3<SPLIT>(co[u], pph, ppl, bh0, bh1, bl0, bl1);
            }
#pragma unroll
            for (int i = 0; i < 2; ++i)
                *reinterpret_cast<float2 *>(sR + (gq + 8 * i) * L.rstride + 8 * nt + 2 * tq) =
                    make_float2(cr[u][2 * i], cr[u][2 * i + 1]);
        }
        __syncthreads();
        // ---------------- U_I by forward substitution through A_II
        if (tid < dvp) {
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) x[r] = sR[r * L.rstride + tid];
#pragma unroll
            for (int r = 1; r < 16; ++r) {
                float acc = x[r];
#pragma unroll
                for (int s2 = 0; s2 < r; ++s2) acc -= sAd[r * 16 + s2] * x[s2];
                x[r] = acc;
            }
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                uint32_t hi, lo;
                pack2<SPLIT>(x[2 * m], x[2 * m + 1], hi, lo);
                const int o = (8 * I + m) * L.ustride + tid;
                sw[L.u + o] = hi;
                if (SPLIT) sw[L.u + lo_u + o] = lo;
            }
        }
        __syncthreads();
        // ---------------- o += P_II U_I, store
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int nt = warp + 8 * u;
            if (nt >= n_nt) break;
            const int col = 8 * nt + gq;
            const uint32_t *f = sFr + I * FW + M * 128;
            uint32_t pph[4], ppl[4];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                pph[x] = f[x * 32 + lane];
                ppl[x] = SPLIT ? f[128 + x * 32 + lane] : 0u;
            }
            const int o0 = (8 * I + tq) * L.ustride + col, o1 = o0 + 4 * L.ustride;
            const uint32_t bh0 = sw[L.u + o0], bh1 = sw[L.u + o1];
            const uint32_t bl0 = SPLIT ? sw[L.u + lo_u + o0] : 0u;
            const uint32_t bl1 = SPLIT ? sw[L.u + lo_u + o1] : 0u;
            mma3<SPLIT>(co[u], pph, ppl, bh0, bh1, bl0, bl1);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int r = gq + 8 * i;
                if (r < nrow)
                    st2(out + ((size_t)b * T + r0 + r) * HV * dv + (size_t)hv * dv + j0 + 8 * nt + 2 * tq,
                        co[u][2 * i], co[u][2 * i + 1]);
            }
        }
        // the next block rewrites the tiles and beta, and its stage buffer
        // (one stage: the one read here)
        __syncthreads();
        if (nstage == 1 && I + 1 < NBT) stage_block(I + 1);
    }
}

// ------------------------------------------------------------------ host side
int tree_pad(int T) { return T <= 32 ? 32 : (T + 31) / 32 * 32; }
size_t align_up(size_t x) { return (x + 255) / 256 * 256; }
constexpr size_t kSmemLimit = 227 * 1024;

// Columns of dv per solve CTA and its fragment stages: one stage when that
// fits a wider part in fewer waves of CTAs, two (the next block's fragments
// copying in during this one) otherwise.
struct TreePart {
    int dvp, nstage;
};
struct TreeLayout {
    int Tp, NBT, NTRI, dkG, m;
    size_t anc, Gp, Gref, spread, Kh, frags, nz, Ad, total;
};
TreeLayout tree_layout_of(const Problem &p) {
    TreeLayout L;
    L.Tp = tree_pad(p.T);
    L.NBT = (p.T + 15) / 16;
    L.NTRI = L.NBT * (L.NBT + 1) / 2;
    L.dkG = p.g_scalar ? 1 : p.dk;
    L.m = p.bf16 ? 1 : 2;
    const size_t trees = (size_t)p.B * p.HV;
    size_t o = 0;
    L.anc = o; o += align_up((size_t)p.B * L.Tp * (L.Tp / 32) * 4);
    L.Gp = o; o += align_up(trees * L.Tp * L.dkG * 4);
    const bool cw = !p.g_scalar;  // block references and column operands: channelwise only
    L.Gref = o; o += cw ? align_up(trees * L.NBT * p.dk * 4) : 0;
    L.spread = o; o += cw ? align_up(trees * L.NBT * (p.dk / kPathCh) * 4) : 0;
    L.Kh = o; o += cw ? align_up(trees * L.Tp * (p.dk / 2) * L.m * 4) : 0;
    L.frags = o; o += align_up(trees * L.NTRI * 2 * L.m * 128 * 4);
    L.nz = o; o += align_up(trees * L.NTRI * 4);
    L.Ad = o; o += align_up(trees * L.NBT * 256 * 4);
    L.total = o;
    return L;
}

template <typename IO, int DK, bool SPLIT, bool SCALAR_G>
cudaError_t launch_solve(const SolveArgs &a, int trees, size_t smem, cudaStream_t s) {
    auto kern = gdr_tree_solve_kernel<IO, DK, SPLIT, SCALAR_G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(a.dv / a.dvp, trees), kTreeThreads, smem, s>>>(a);
    return cudaGetLastError();
}
template <typename IO, int DK, bool SPLIT, bool SCALAR_G, bool PER_KH>
cudaError_t launch_gram(const GramArgs &a, int B, size_t smem, cudaStream_t s) {
    auto kern = gdr_tree_gram_kernel<IO, DK, SPLIT, SCALAR_G, PER_KH>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(a.NBT, B * (PER_KH ? a.HK : a.HV)), kTreeThreads, smem, s>>>(a);
    return cudaGetLastError();
}

template <typename IO, int DK, bool SPLIT>
cudaError_t launch_tree_kernels(const Problem &p, const GramArgs &ga, const SolveArgs &sa,
                                bool per_kh, cudaStream_t s) {
    const bool h0 = p.h0 != nullptr;
    const size_t gsmem = (size_t)gram_smem_words(ga.Tp, DK, SPLIT, per_kh ? p.HV / p.HK : 1) * 4;
    const size_t ssmem = (size_t)solve_smem(sa.Tp, sa.NBT, DK, sa.dvp, SPLIT, h0, sa.nstage).words * 4;
    cudaError_t e;
    trace_begin(kKernTreeGram, s);
    if (p.g_scalar)
        e = per_kh ? launch_gram<IO, DK, SPLIT, true, true>(ga, p.B, gsmem, s)
                   : launch_gram<IO, DK, SPLIT, true, false>(ga, p.B, gsmem, s);
    else
        e = launch_gram<IO, DK, SPLIT, false, false>(ga, p.B, gsmem, s);
    if (e != cudaSuccess) return e;
    trace_end(kKernTreeGram, s);
    trace_begin(kKernTreeSolve, s);
    e = p.g_scalar ? launch_solve<IO, DK, SPLIT, true>(sa, p.B * p.HV, ssmem, s)
                   : launch_solve<IO, DK, SPLIT, false>(sa, p.B * p.HV, ssmem, s);
    if (e != cudaSuccess) return e;
    trace_end(kKernTreeSolve, s);
    return cudaSuccess;
}
template <typename IO, bool SPLIT>
cudaError_t launch_tree_dk(const Problem &p, const GramArgs &ga, const SolveArgs &sa, bool per_kh,
                           cudaStream_t s) {
    switch (p.dk) {
        case 32: return launch_tree_kernels<IO, 32, SPLIT>(p, ga, sa, per_kh, s);
        case 64: return launch_tree_kernels<IO, 64, SPLIT>(p, ga, sa, per_kh, s);
        case 128: return launch_tree_kernels<IO, 128, SPLIT>(p, ga, sa, per_kh, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

// Columns of dv per solve CTA: the widest part whose shared memory fits,
// then narrower while twice the CTAs still fit on the device at once (the
// walk over the blocks is serial: more CTAs in flight is more of it in
// parallel).
static TreePart tree_part_choice(const Problem &p) {
    const int Tp = tree_pad(p.T), NBT = (p.T + 15) / 16;
    const bool split = p.bf16 == 0, h0 = p.h0 != nullptr;
    auto bytes = [&](int dvp, int ns) {
        return (size_t)solve_smem(Tp, NBT, p.dk, dvp, split, h0, ns).words * 4;
    };
    auto widest = [&](int ns) {
        int dvp = p.dv;
        while (dvp > 16 && bytes(dvp, ns) > kSmemLimit) dvp /= 2;
        return bytes(dvp, ns) <= kSmemLimit ? dvp : 0;
    };
    int sms = 148, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    auto waves = [&](int dvp, int ns) {
        const long long per_sm = std::min<long long>(2, (long long)(kSmemLimit / bytes(dvp, ns)));
        const long long ctas = (long long)p.B * p.HV * (p.dv / dvp);
        return (ctas + sms * per_sm - 1) / (sms * per_sm);
    };
    TreePart t{widest(2), 2};
    const int w1 = widest(1);
    if (w1 == 0) return TreePart{0, 1};
    if (t.dvp == 0 || waves(w1, 1) < waves(t.dvp, 2)) t = TreePart{w1, 1};
    // narrower while twice the CTAs still fit on the device at once (the walk
    // over the blocks is serial: more CTAs in flight is more of it in parallel)
    while (t.dvp >= 64 && bytes(t.dvp / 2, t.nstage) <= kSmemLimit && waves(t.dvp / 2, t.nstage) <= 1 &&
           waves(t.dvp, t.nstage) <= 1)
        t.dvp /= 2;
    return t;
}
int tree_blocked_part(const Problem &p) { return tree_part_choice(p).dvp; }

bool tree_blocked_supported(const Problem &p) {
    return p.T >= 1 && p.T <= kTreeMaxT && (p.dk == 32 || p.dk == 64 || p.dk == 128) &&
           p.dv % 32 == 0 && tree_blocked_part(p) > 0;
}

size_t tree_blocked_workspace_bytes(const Problem &p) { return tree_layout_of(p).total; }

cudaError_t launch_tree_blocked(const Problem &p, void *workspace, const int *parents,
                                unsigned variant, cudaStream_t stream) {
    const TreeLayout L = tree_layout_of(p);
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    uint32_t *anc = reinterpret_cast<uint32_t *>(ws + L.anc);
    float *Gp = reinterpret_cast<float *>(ws + L.Gp);
    int rounds = 0;
    while ((1 << rounds) < p.T) ++rounds;
    cudaError_t e;
    trace_begin(kKernTreePath, stream);
    gdr_tree_mask_kernel<<<p.B, L.Tp, 0, stream>>>(parents, anc, p.T, L.Tp, rounds);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    float *Gref = reinterpret_cast<float *>(ws + L.Gref);
    int *spread = reinterpret_cast<int *>(ws + L.spread);
    uint32_t *Kh = reinterpret_cast<uint32_t *>(ws + L.Kh);
    const dim3 pgrid(p.g_scalar ? 1 : p.dk / kPathCh, p.B * p.HV);
    if (p.g_scalar)
        gdr_tree_path_kernel<float, 1, false><<<pgrid, L.Tp, 0, stream>>>(
            parents, p.g, nullptr, Gp, nullptr, nullptr, nullptr, p.T, L.Tp, L.NBT, p.HK, p.HV, 1, rounds);
    else if (p.bf16)
        gdr_tree_path_kernel<__nv_bfloat16, kPathCh, false><<<pgrid, L.Tp, 0, stream>>>(
            parents, p.g, static_cast<const __nv_bfloat16 *>(p.k), Gp, Gref, spread, Kh, p.T, L.Tp,
            L.NBT, p.HK, p.HV, p.dk, rounds);
    else
        gdr_tree_path_kernel<float, kPathCh, true><<<pgrid, L.Tp, 0, stream>>>(
            parents, p.g, static_cast<const float *>(p.k), Gp, Gref, spread, Kh, p.T, L.Tp, L.NBT,
            p.HK, p.HV, p.dk, rounds);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    trace_end(kKernTreePath, stream);

    GramArgs ga;
    ga.q = p.q; ga.k = p.k; ga.beta = p.beta; ga.Gp = Gp; ga.anc = anc;
    ga.Gref = Gref; ga.spread = spread; ga.Kh = Kh;
    ga.frags = reinterpret_cast<uint32_t *>(ws + L.frags);
    ga.nz = reinterpret_cast<int *>(ws + L.nz);
    ga.Ad = reinterpret_cast<float *>(ws + L.Ad);
    ga.T = p.T; ga.Tp = L.Tp; ga.NBT = L.NBT; ga.HK = p.HK; ga.HV = p.HV;
    SolveArgs sa;
    sa.q = p.q; sa.k = p.k; sa.v = p.v; sa.beta = p.beta; sa.h0 = p.h0; sa.out = p.out;
    sa.Gp = Gp; sa.frags = ga.frags; sa.nz = ga.nz; sa.Ad = ga.Ad;
    sa.T = p.T; sa.Tp = L.Tp; sa.NBT = L.NBT; sa.HK = p.HK; sa.HV = p.HV; sa.dv = p.dv;
    const TreePart part = tree_part_choice(p);
    sa.dvp = part.dvp;
    sa.nstage = part.nstage;
    if (sa.dvp <= 0) return cudaErrorInvalidValue;
    // the gram per key head only where it saves work: a scalar gate, and
    // value heads sharing a key head
    const bool per_kh = p.g_scalar && p.HV > p.HK && !(variant & kTreeGramPerValueHead);
    if (p.bf16) return launch_tree_dk<__nv_bfloat16, false>(p, ga, sa, per_kh, stream);
    return launch_tree_dk<float, true>(p, ga, sa, per_kh, stream);
}

}  // namespace gdr
