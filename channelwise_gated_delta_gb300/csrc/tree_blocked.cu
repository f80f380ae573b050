// tree_blocked.cu -- tree verification of up to 512 draft tokens: the whole
// tree as one unit-lower system, solved 16 rows at a time.
//
// Page "Support TreeUpdateSolve kernel" (trymirai/uzu PR #576), commit
// summary: a gram of block pairs, 16 x 16 diagonal blocks, and a block
// forward substitution (a "pure block TRSM") whose right-hand side starts
// from kh0 = the decayed keys against h0.  Page "Reorder channelwise gated
// delta rule chunked hot loops" (pytorch/executorch): the chunkwise WY form,
// here over a tree's ancestor relation instead of the causal order.
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
// Launches:
//  gdr_tree_path_kernel     G (log2 units) and the strict-ancestor bitmasks,
//                           by pointer jumping (ceil(log2 T) rounds);
//  gdr_tree_blocked_kernel  one CTA per (tree, value head, dv part) walks the
//                           16-row blocks I in order: grams A_IJ, P_IJ (J <= I,
//                           block pairs with no ancestor pair skipped) on bf16
//                           mma.sync, the right-hand side from kh0 and the
//                           earlier blocks' U, U_I by forward substitution
//                           through A_II in f32, then o.
// Decay factors of a block pair are split about a per-channel reference, the
// largest G over the row block's tokens: row operands take exp(G_r - Gref)
// <= 1, column operands exp(Gref - G_s), which for an ancestor s of a row of
// the block is at most the block's spread max_r (Gref - G_r).  A row block
// spread over more than 60 nats runs one pass per row instead, each row its
// own reference (column factors <= 1).  f32 q/k/v carry every tensor-core
// operand as a bf16 pair hi + lo and every product as hi hi + hi lo + lo hi
// (BF16x3); bf16 q/k/v use one bf16 product.
#include <string.h>

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

// ------------------------------------------------------------------ path kernel
// grid (ngroups + 1, B * HV).  x < ngroups: channels [32 x, 32 x + CH) of
// G for tree (b, hv); x == ngroups (hv == 0 only): the ancestor masks of b.
__global__ void __launch_bounds__(kTreeThreads)
    gdr_tree_path_kernel(const int *__restrict__ parent, const float *__restrict__ g,
                         float *__restrict__ Gp, uint32_t *__restrict__ anc, int T, int Tp, int HV,
                         int dkG, int ngroups, int rounds) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int tree = blockIdx.y, b = tree / HV, hv = tree % HV, tid = threadIdx.x;
    int *P0 = reinterpret_cast<int *>(smem_raw);
    int *P1 = P0 + Tp;
    for (int t = tid; t < Tp; t += kTreeThreads) P0[t] = t < T ? parent[(size_t)b * T + t] : -1;
    __syncthreads();  // every parent in place before any thread follows one
    if ((int)blockIdx.x < ngroups) {
        const int c0 = 32 * blockIdx.x, CH = min(32, dkG - c0);
        float *G0 = reinterpret_cast<float *>(P1 + Tp);
        float *G1 = G0 + Tp * CH;
        for (int idx = tid; idx < Tp * CH; idx += kTreeThreads) {
            const int t = idx / CH, c = idx - t * CH;
            G0[idx] = t < T ? g[((size_t)b * T + t) * HV * dkG + (size_t)hv * dkG + c0 + c] * kLog2eT
                            : 0.f;
        }
        __syncthreads();
        for (int r = 0; r < rounds; ++r) {
            for (int idx = tid; idx < Tp * CH; idx += kTreeThreads) {
                const int t = idx / CH, c = idx - t * CH, p = P0[t];
                G1[idx] = G0[idx] + (p >= 0 ? G0[p * CH + c] : 0.f);
            }
            for (int t = tid; t < Tp; t += kTreeThreads) {
                const int p = P0[t];
                P1[t] = p >= 0 ? P0[p] : -1;
            }
            __syncthreads();
            float *gt = G0; G0 = G1; G1 = gt;
            int *pt = P0; P0 = P1; P1 = pt;
        }
        for (int idx = tid; idx < Tp * CH; idx += kTreeThreads) {
            const int t = idx / CH, c = idx - t * CH;
            Gp[((size_t)tree * Tp + t) * dkG + c0 + c] = G0[idx];
        }
    } else if (hv == 0) {
        const int NW = Tp / 32;
        uint32_t *M0 = reinterpret_cast<uint32_t *>(P1 + Tp);
        uint32_t *M1 = M0 + Tp * NW;
        for (int idx = tid; idx < Tp * NW; idx += kTreeThreads) {
            const int t = idx / NW, w = idx - t * NW, p = P0[t];
            M0[idx] = (p >= 0 && (p >> 5) == w) ? (1u << (p & 31)) : 0u;
        }
        __syncthreads();
        for (int r = 0; r < rounds; ++r) {
            for (int idx = tid; idx < Tp * NW; idx += kTreeThreads) {
                const int t = idx / NW, w = idx - t * NW, p = P0[t];
                M1[idx] = M0[idx] | (p >= 0 ? M0[p * NW + w] : 0u);
            }
            for (int t = tid; t < Tp; t += kTreeThreads) {
                const int p = P0[t];
                P1[t] = p >= 0 ? P0[p] : -1;
            }
            __syncthreads();
            uint32_t *mt = M0; M0 = M1; M1 = mt;
            int *pt = P0; P0 = P1; P1 = pt;
        }
        for (int idx = tid; idx < Tp * NW; idx += kTreeThreads) anc[(size_t)b * Tp * NW + idx] = M0[idx];
    }
}

// ------------------------------------------------------------------ main kernel
struct TreeArgs {
    const void *q, *k, *v;
    const float *beta, *h0;
    void *out;
    const float *Gp;      // [B * HV][Tp][dk or 1] path prefix sums, log2 units
    const uint32_t *anc;  // [B][Tp][Tp / 32] strict-ancestor bitmasks
    int T, Tp, HK, HV, dv, dvp;
};

// Shared-memory map (32-bit words), sized by Tp, dk, dvp; "hi" arrays are
// followed by their "lo" halves when SPLIT.
struct TreeSmem {
    int u, ustride;    // U history: [Tp / 2][ustride] bf16 row pairs
    int afr, pfr;      // -A and P block fragments: [NB][4][32]
    int ad;            // f32 A_II [16][17]
    int h0, hstride;   // h0 part: [dk / 2][hstride] bf16 channel pairs
    int lk, lq, lk0, lq0, tstride;  // row tiles [16][tstride]
    int r, rstride;    // f32 right-hand side [16][rstride] (over lk0 / lq0)
    int gref, grow, mask, beta, nz, flag;
    int words;
};
__host__ __device__ inline TreeSmem tree_smem(int Tp, int dk, int dvp, bool split) {
    TreeSmem s;
    const int m = split ? 2 : 1, NB = Tp / 16;
    int o = 0;
    s.ustride = dvp + 8;
    s.u = o; o += m * (Tp / 2) * s.ustride;
    s.afr = o; o += m * NB * 128;
    s.pfr = o; o += m * NB * 128;
    s.ad = o; o += 16 * 17;
    s.hstride = dvp + 8;
    s.h0 = o; o += m * (dk / 2) * s.hstride;
    s.tstride = dk / 2 + 4;
    const int tile = m * 16 * s.tstride;
    s.lk = o; o += tile;
    s.lq = o; o += tile;
    s.rstride = dvp + 4;
    s.lk0 = o;
    s.lq0 = o + tile;
    s.r = o;
    o += max(2 * tile, 16 * s.rstride);
    s.gref = o; o += dk;
    s.grow = o; o += 16;
    s.mask = o; o += 16 * (Tp / 32);
    s.beta = o; o += 16;
    s.nz = o; o += NB;
    s.flag = o; o += 4;
    s.words = o;
    return s;
}

template <typename IO, int DK, bool SPLIT, bool SCALAR_G>
__global__ void __launch_bounds__(kTreeThreads, 1) gdr_tree_blocked_kernel(const TreeArgs a) {
    extern __shared__ __align__(16) uint32_t sw[];
    const int Tp = a.Tp, T = a.T, NB = (T + 15) / 16, NW = Tp / 32;
    const TreeSmem L = tree_smem(Tp, DK, a.dvp, SPLIT);
    const int tree = blockIdx.y, HV = a.HV, b = tree / HV, hv = tree % HV;
    const int hk = hv / (HV / a.HK);
    const int j0 = blockIdx.x * a.dvp, dvp = a.dvp, dv = a.dv;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3;
    const IO *q = static_cast<const IO *>(a.q);
    const IO *k = static_cast<const IO *>(a.k);
    const IO *v = static_cast<const IO *>(a.v);
    IO *out = static_cast<IO *>(a.out);
    constexpr int DKG = SCALAR_G ? 1 : DK;
    const float *Gt = a.Gp + (size_t)tree * Tp * DKG;  // this tree's G
    const uint32_t *ancb = a.anc + (size_t)b * Tp * NW;
    const int lo_u = (Tp / 2) * L.ustride, lo_fr = NB * 128, lo_h = (DK / 2) * L.hstride,
              lo_t = 16 * L.tstride;
    float *sR = reinterpret_cast<float *>(sw + L.r);
    float *sAd = reinterpret_cast<float *>(sw + L.ad);
    float *sGref = reinterpret_cast<float *>(sw + L.gref);
    float *sGrow = reinterpret_cast<float *>(sw + L.grow);
    float *sBeta = reinterpret_cast<float *>(sw + L.beta);
    uint32_t *sMask = sw + L.mask;
    int *sNz = reinterpret_cast<int *>(sw + L.nz);
    const bool has_h0 = a.h0 != nullptr;
    auto krow = [&](int t) { return k + ((size_t)b * T + t) * a.HK * DK + (size_t)hk * DK; };
    auto qrow = [&](int t) { return q + ((size_t)b * T + t) * a.HK * DK + (size_t)hk * DK; };

    // h0 part as bf16 channel pairs (hi, lo)
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
    const int n_nt = dvp / 8;  // n-tiles of this part; warp w owns w and w + 8

#pragma unroll 1
    for (int I = 0; I < NB; ++I) {
        const int r0 = 16 * I, nrow = min(16, T - r0);
        // ---------------- stage 1: the block's rows
        if (tid < 16) {
            sBeta[tid] = tid < nrow ? a.beta[((size_t)b * T + r0 + tid) * HV + hv] : 0.f;
            if (SCALAR_G) sGrow[tid] = tid < nrow ? Gt[r0 + tid] : 0.f;
        }
        for (int idx = tid; idx < 16 * NW; idx += kTreeThreads) {
            const int r = idx / NW;
            sMask[idx] = r < nrow ? ancb[(size_t)r0 * NW + idx] : 0u;
        }
        int bad = 0;
        if (!SCALAR_G) {
            for (int c = tid; c < DK; c += kTreeThreads) {
                float m = -3.0e38f, lo = 3.0e38f;
                for (int r = 0; r < nrow; ++r) {
                    const float x = Gt[(size_t)(r0 + r) * DK + c];
                    m = fmaxf(m, x);
                    lo = fminf(lo, x);
                }
                sGref[c] = m;
                bad |= !(m - lo <= kSpreadLog2);
            }
        }
        const bool fallback = __syncthreads_or(bad) != 0;
        for (int idx = tid; idx < 16 * (DK / 2); idx += kTreeThreads) {
            const int r = idx / (DK / 2), cp = idx - r * (DK / 2), c = 2 * cp;
            float2 kk = make_float2(0.f, 0.f), qq = kk, e = make_float2(1.f, 1.f), e0 = e;
            if (r < nrow) {
                kk = ld2(krow(r0 + r) + c);
                qq = ld2(qrow(r0 + r) + c);
                if (SCALAR_G) {
                    const float x = ex2(Gt[r0 + r]);
                    e0 = make_float2(x, x);
                } else {
                    const float2 gg = *reinterpret_cast<const float2 *>(Gt + (size_t)(r0 + r) * DK + c);
                    e = make_float2(ex2(gg.x - sGref[c]), ex2(gg.y - sGref[c + 1]));
                    e0 = make_float2(ex2(gg.x), ex2(gg.y));
                }
            }
            uint32_t hi, lo;
            const int o = r * L.tstride + cp;
            pack2<SPLIT>(kk.x * e.x, kk.y * e.y, hi, lo);
            sw[L.lk + o] = hi;
            if (SPLIT) sw[L.lk + lo_t + o] = lo;
            pack2<SPLIT>(qq.x * e.x, qq.y * e.y, hi, lo);
            sw[L.lq + o] = hi;
            if (SPLIT) sw[L.lq + lo_t + o] = lo;
            if (has_h0) {
                pack2<SPLIT>(kk.x * e0.x, kk.y * e0.y, hi, lo);
                sw[L.lk0 + o] = hi;
                if (SPLIT) sw[L.lk0 + lo_t + o] = lo;
                pack2<SPLIT>(qq.x * e0.x, qq.y * e0.y, hi, lo);
                sw[L.lq0 + o] = hi;
                if (SPLIT) sw[L.lq0 + lo_t + o] = lo;
            }
        }
        __syncthreads();
        // ---------------- stage 2: grams A_IJ, P_IJ (warp per block pair)
#pragma unroll 1
        for (int J = warp; J <= I; J += kTreeThreads / 32) {
            // ancestor bits of this lane's rows gq, gq + 8 among the columns of J
            const int sh = 16 * (J & 1);
            const uint32_t f0 = (sMask[gq * NW + (J >> 1)] >> sh) & 0xffffu;
            const uint32_t f1 = (sMask[(gq + 8) * NW + (J >> 1)] >> sh) & 0xffffu;
            const bool any = __any_sync(0xffffffffu, (f0 | f1) != 0u) || J == I;
            if (lane == 0) sNz[J] = any ? 1 : 0;
            if (!any) continue;
            float ca[2][4], cp[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) ca[nt][e] = cp[nt][e] = 0.f;
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
                            const int o = (gq + 8 * (x & 1)) * L.tstride + 8 * ks + tq + 4 * (x >> 1);
                            akh[x] = sw[L.lk + o];
                            aqh[x] = sw[L.lq + o];
                            akl[x] = SPLIT ? sw[L.lk + lo_t + o] : 0u;
                            aql[x] = SPLIT ? sw[L.lq + lo_t + o] : 0u;
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
            // epilogue: ancestor mask, beta, scalar decays; fragments of -A and P
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
                            const float d = ex2(fminf(sGrow[r] - Gt[16 * J + sl], 0.f));
                            x *= d;
                            y *= d;
                        }
                        va[e] = an ? sBeta[r] * x : 0.f;
                        vp[e] = (an || self) ? y : 0.f;
                        if (J == I) sAd[r * 17 + sl] = va[e];
                    }
                    const int reg = 2 * nt + i, o = (J * 4 + reg) * 32 + lane;
                    uint32_t hi, lo;
                    pack2<SPLIT>(-va[0], -va[1], hi, lo);
                    sw[L.afr + o] = hi;
                    if (SPLIT) sw[L.afr + lo_fr + o] = lo;
                    pack2<SPLIT>(vp[0], vp[1], hi, lo);
                    sw[L.pfr + o] = hi;
                    if (SPLIT) sw[L.pfr + lo_fr + o] = lo;
                }
            }
        }
        __syncthreads();
        // ---------------- stage 3: right-hand side and output from h0 and the earlier blocks
        float cr[2][4], co[2][4];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int nt = warp + 8 * u;
            if (nt >= n_nt) break;
#pragma unroll
            for (int e = 0; e < 4; ++e) cr[u][e] = co[u][e] = 0.f;
            const int col = 8 * nt + gq;
            if (has_h0) {
#pragma unroll 2
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
            // rhs = beta_r (v_r - kh0_r)
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int r = gq + 8 * i;
                float2 vv = make_float2(0.f, 0.f);
                if (r < nrow)
                    vv = ld2(v + ((size_t)b * T + r0 + r) * HV * dv + (size_t)hv * dv + j0 + 8 * nt + 2 * tq);
                cr[u][2 * i] = sBeta[r] * (vv.x - cr[u][2 * i]);
                cr[u][2 * i + 1] = sBeta[r] * (vv.y - cr[u][2 * i + 1]);
            }
#pragma unroll 1
            for (int J = 0; J < I; ++J) {
                if (!sNz[J]) continue;
                uint32_t aah[4], aal[4], pph[4], ppl[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const int o = (J * 4 + x) * 32 + lane;
                    aah[x] = sw[L.afr + o];
                    pph[x] = sw[L.pfr + o];
                    aal[x] = SPLIT ? sw[L.afr + lo_fr + o] : 0u;
                    ppl[x] = SPLIT ? sw[L.pfr + lo_fr + o] : 0u;
                }
                const int o0 = (8 * J + tq) * L.ustride + col, o1 = o0 + 4 * L.ustride;
                const uint32_t bh0 = sw[L.u + o0], bh1 = sw[L.u + o1];
                const uint32_t bl0 = SPLIT ? sw[L.u + lo_u + o0] : 0u;
                const uint32_t bl1 = SPLIT ? sw[L.u + lo_u + o1] : 0u;
                mma3<SPLIT>(cr[u], aah, aal, bh0, bh1, bl0, bl1);
                mma3<SPLIT>(co[u], pph, ppl, bh0, bh1, bl0, bl1);
            }
        }
        __syncthreads();  // the h0 row tiles are read: the rhs goes over them
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int nt = warp + 8 * u;
            if (nt >= n_nt) break;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int r = gq + 8 * i;
                *reinterpret_cast<float2 *>(sR + r * L.rstride + 8 * nt + 2 * tq) =
                    make_float2(cr[u][2 * i], cr[u][2 * i + 1]);
            }
        }
        __syncthreads();
        // ---------------- stage 4: U_I by forward substitution through A_II
        if (tid < dvp) {
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) x[r] = sR[r * L.rstride + tid];
#pragma unroll
            for (int r = 1; r < 16; ++r) {
                float acc = x[r];
#pragma unroll
                for (int s = 0; s < r; ++s) acc -= sAd[r * 17 + s] * x[s];
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
        // ---------------- stage 5: o += P_II U_I, store
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int nt = warp + 8 * u;
            if (nt >= n_nt) break;
            const int col = 8 * nt + gq;
            uint32_t pph[4], ppl[4];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const int o = (I * 4 + x) * 32 + lane;
                pph[x] = sw[L.pfr + o];
                ppl[x] = SPLIT ? sw[L.pfr + lo_fr + o] : 0u;
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
        // the next block's stage 1 rewrites the row tiles, read here no more
        __syncthreads();
    }
}

size_t path_smem_bytes(int Tp, int dkG) {
    const size_t ints = 2 * (size_t)Tp * sizeof(int);
    const size_t g = 2 * (size_t)Tp * min(32, dkG) * sizeof(float);
    const size_t m = 2 * (size_t)Tp * (Tp / 32) * sizeof(uint32_t);
    return ints + (g > m ? g : m);
}

template <typename IO, int DK, bool SPLIT, bool SCALAR_G>
cudaError_t launch_blocked(const TreeArgs &a, int B, size_t smem, cudaStream_t s) {
    auto kern = gdr_tree_blocked_kernel<IO, DK, SPLIT, SCALAR_G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.dv / a.dvp, B * a.HV);
    kern<<<grid, kTreeThreads, smem, s>>>(a);
    return cudaGetLastError();
}

template <typename IO, bool SPLIT, bool SCALAR_G>
cudaError_t launch_blocked_dk(const TreeArgs &a, int B, int dk, size_t smem, cudaStream_t s) {
    switch (dk) {
        case 32: return launch_blocked<IO, 32, SPLIT, SCALAR_G>(a, B, smem, s);
        case 64: return launch_blocked<IO, 64, SPLIT, SCALAR_G>(a, B, smem, s);
        case 128: return launch_blocked<IO, 128, SPLIT, SCALAR_G>(a, B, smem, s);
        default: return cudaErrorInvalidValue;
    }
}

int tree_pad(int T) { return T <= 32 ? 32 : (T + 31) / 32 * 32; }

}  // namespace

// Columns of dv per CTA: the widest part whose shared memory fits.
int tree_blocked_part(const Problem &p) {
    const int Tp = tree_pad(p.T);
    for (int dvp = p.dv; dvp >= 16; dvp /= 2) {
        const TreeSmem s = tree_smem(Tp, p.dk, dvp, p.bf16 == 0);
        if ((size_t)s.words * 4 <= 227 * 1024) return dvp;
    }
    return 0;
}

bool tree_blocked_supported(const Problem &p) {
    return p.T >= 1 && p.T <= kTreeMaxT && (p.dk == 32 || p.dk == 64 || p.dk == 128) &&
           p.dv % 32 == 0 && tree_blocked_part(p) > 0;
}

size_t tree_blocked_workspace_bytes(const Problem &p) {
    const int Tp = tree_pad(p.T);
    const size_t dkG = p.g_scalar ? 1 : (size_t)p.dk;
    const size_t anc = (size_t)p.B * Tp * (Tp / 32) * sizeof(uint32_t);
    const size_t G = (size_t)p.B * p.HV * Tp * dkG * sizeof(float);
    return ((anc + 255) / 256 * 256) + ((G + 255) / 256 * 256);
}

cudaError_t launch_tree_blocked(const Problem &p, void *workspace, const int *parents,
                                cudaStream_t stream) {
    const int Tp = tree_pad(p.T);
    const int dkG = p.g_scalar ? 1 : p.dk;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    uint32_t *anc = reinterpret_cast<uint32_t *>(ws);
    const size_t anc_bytes = (size_t)p.B * Tp * (Tp / 32) * sizeof(uint32_t);
    float *Gp = reinterpret_cast<float *>(ws + (anc_bytes + 255) / 256 * 256);
    int rounds = 0;
    while ((1 << rounds) < p.T) ++rounds;
    const int ngroups = (dkG + 31) / 32;
    const size_t psmem = path_smem_bytes(Tp, dkG);
    cudaError_t e = cudaFuncSetAttribute(gdr_tree_path_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)psmem);
    if (e != cudaSuccess) return e;
    trace_begin(kKernTreePath, stream);
    gdr_tree_path_kernel<<<dim3(ngroups + 1, p.B * p.HV), kTreeThreads, psmem, stream>>>(
        parents, p.g, Gp, anc, p.T, Tp, p.HV, dkG, ngroups, rounds);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    trace_end(kKernTreePath, stream);

    TreeArgs a;
    a.q = p.q; a.k = p.k; a.v = p.v; a.beta = p.beta; a.h0 = p.h0; a.out = p.out;
    a.Gp = Gp; a.anc = anc;
    a.T = p.T; a.Tp = Tp; a.HK = p.HK; a.HV = p.HV; a.dv = p.dv;
    a.dvp = tree_blocked_part(p);
    const bool split = p.bf16 == 0;
    const size_t smem = (size_t)tree_smem(Tp, p.dk, a.dvp, split).words * 4;
    trace_begin(kKernTreeBlocked, stream);
    if (p.bf16) {
        e = p.g_scalar ? launch_blocked_dk<__nv_bfloat16, false, true>(a, p.B, p.dk, smem, stream)
                       : launch_blocked_dk<__nv_bfloat16, false, false>(a, p.B, p.dk, smem, stream);
    } else {
        e = p.g_scalar ? launch_blocked_dk<float, true, true>(a, p.B, p.dk, smem, stream)
                       : launch_blocked_dk<float, true, false>(a, p.B, p.dk, smem, stream);
    }
    if (e != cudaSuccess) return e;
    trace_end(kKernTreeBlocked, stream);
    return cudaSuccess;
}

}  // namespace gdr
