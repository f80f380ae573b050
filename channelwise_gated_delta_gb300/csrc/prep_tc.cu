// prep_tc.cu -- the per-chunk preparation of the chunked prefill on the
// tensor cores (dk = dv = 128, chunk 64): the records the tensor-core state
// scan (scan_tc.cu) reads, built with tcgen05 products accumulated in tensor
// memory instead of warp-level mma.sync.
//
// Page "Reorder channelwise gated delta rule chunked hot loops for
// autovectorization" (pytorch/executorch PR #21021), second commit summary:
// per chunk the per-channel log-decay prefix sums, the causal key/key and
// query/key terms, the beta-folded unit-lower transform and the WY
// pseudo-keys and pseudo-values.  With G the inclusive prefix sum of g over
// the chunk, m its middle row and L its length:
//   Lk = K e^{G - G_m},  Lq = Q e^{G - G_m},  R = K e^{G_m - G}
//   A = tril(diag(beta) Lk R^T, -1),  P = tril(Lq R^T)
//   T = (I + A)^-1,  Wk = T diag(beta) (K e^G),  Wv = T diag(beta) V
//   Qt = Q e^G,  Kh = K e^{G_L - G},  gam = e^{G_L}
// (the factors of Lk, Lq and R meet in each product, so A and P hold the
// exact decays e^{G_r - G_s}).
//
// One CTA per (chunk, value head), sixteen warps:
//   1. prefix sums (one thread per key channel) into shared memory;
//   2. the operand tiles, eight channels of one row per thread: [Lk; Lq] and
//      R as bf16 hi/lo pairs for the gram, diag(beta) K e^G for the WY
//      product, and the Qt and Kh records straight to global memory;
//   3. one M = 128 gram [Lk; Lq] R^T (BF16x3: hi.hi + hi.lo + lo.hi, f32
//      accumulation in tensor memory) while the threads build diag(beta) V;
//   4. A (tensor-memory lanes 0-63) into shared memory, P (lanes 64-127)
//      into its record;
//   5. T by blocks of 16 on CUDA cores in f32: the diagonal blocks by
//      forward substitution, then T_IJ = -T_II sum_K A_IK T_KJ level by level;
//   6. W = T [diag(beta) K e^G | diag(beta) V] as two M = 128, N = 128
//      products (BF16x3; rows 64-127 of the A operand are not used);
//   7. Wk and Wv out of tensor memory into their records.
// A chunk whose factors would leave e^{+-60} (strong decay) takes A and P
// from the pairwise decays instead (every exponent <= 0), on CUDA cores.
//
// Records: the layout gdr_chunk_prep writes for the tensor-core scan (Wk,
// Qt, Kh, P as bf16 hi | lo tiles in the K-major interleaved order, Wv f32,
// gam f32).  Every wait is bounded: a timeout sets the library's error word
// and the CTA skips the rest.
#include "common.cuh"
#include "sm100_ptx.cuh"

namespace gdr {
namespace {

using namespace sm100;

constexpr int kPtThreads = 512;
constexpr int kPtWarps = kPtThreads / 32;
constexpr int kPtItems = 64 * 16 / kPtThreads;  // (row, 8-channel octet) items a thread
constexpr int kPtC = 64;   // chunk
constexpr int kPtD = 128;  // dk = dv
constexpr uint64_t kPtWaitNs = 2000000000ull;
// largest log-decay span a factor of the reference-row split may carry:
// e^{-60} keeps the lo part of a bf16 pair a normal number
constexpr float kPtRange = 60.f;
constexpr float kLog2e = 1.4426950408889634f;

// shared memory (bytes from a 1024-byte aligned base)
constexpr uint32_t kPtAop = 0;         // [Lk; Lq] hi | lo, [128 rows][128 k] bf16 K-major
constexpr uint32_t kPtR = 65536;       // R hi | lo, [64][128]
constexpr uint32_t kPtRk = 98304;      // diag(beta) K e^G hi | lo, [64 s][128 i] (read MN-major)
constexpr uint32_t kPtGs = 131072;     // G f32 [64][kPtLdg]; then diag(beta) V hi | lo
constexpr int kPtLdg = 132;
constexpr uint32_t kPtVec = kPtGs + 64 * kPtLdg * 4;  // beta [64], G_m [128], G_L [128], G_31 [128]
constexpr uint32_t kPtBars = kPtVec + 448 * 4;
constexpr uint32_t kPtSlot = kPtBars + 64;
constexpr uint32_t kPtAbort = kPtSlot + 4;
constexpr uint32_t kPtSmem = kPtAbort + 4 + 1024;  // + alignment slack
// after the gram, inside the [Lk; Lq] region
constexpr uint32_t kPtAs = 0;          // A f32 [64][kPtLda]
constexpr int kPtLda = 68;
constexpr uint32_t kPtTf = 17408;      // T f32 [64][kPtLda] (the exact path stages P here first)
constexpr uint32_t kPtX = 34816;       // X blocks f32 [3][16][16]
constexpr uint32_t kPtT = 40960;       // T hi | lo [64][64] bf16 K-major (8 KB each)
// the exact path's transposed copies (channel-major [128][64] f32)
constexpr uint32_t kPtKT = kPtR;       // K^T
constexpr uint32_t kPtQT = 32768;      // Q^T (upper half of the [Lk; Lq] region)
static_assert(kPtT + 3 * 8192 <= 65536, "the T operand's 128 rows stay in the region");
static_assert(kPtX + 3 * 256 * 4 <= kPtT, "X blocks below T");
static_assert(kPtGs + 32768 <= kPtVec, "diag(beta) V fits where G was");

struct PrepTcArgs {
    const void *q, *k, *v;
    const float *g, *beta;
    float *ws;            // records
    const int2 *chunks;   // packed batches: {first row, length} per chunk, or null
    int *err;
    int T, HK, HV, NC, g_scalar;
    size_t rec_floats;
};

// bf16 pair of x: hi = bf16(x), lo = bf16(x - hi)
__device__ __forceinline__ void pt_split(float a, float b, uint32_t &hi, uint32_t &lo) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    hi = *reinterpret_cast<uint32_t *>(&h);
    const float2 f = __bfloat1622float2(h);
    __nv_bfloat162 l = __floats2bfloat162_rn(a - f.x, b - f.y);
    lo = *reinterpret_cast<uint32_t *>(&l);
}
// eight values as the hi and lo 16-byte rows of a core matrix
__device__ __forceinline__ void pt_split8(const float (&x)[8], uint4 &hi, uint4 &lo) {
    pt_split(x[0], x[1], hi.x, lo.x);
    pt_split(x[2], x[3], hi.y, lo.y);
    pt_split(x[4], x[5], hi.z, lo.z);
    pt_split(x[6], x[7], hi.w, lo.w);
}
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
__device__ __forceinline__ void pt_load8(const float *p, float (&x)[8]) {
    const float4 a = *reinterpret_cast<const float4 *>(p);
    const float4 b = *reinterpret_cast<const float4 *>(p + 4);
    x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = b.x, x[5] = b.y, x[6] = b.z, x[7] = b.w;
}
__device__ __forceinline__ void pt_load8(const __nv_bfloat16 *p, float (&x)[8]) {
    const uint4 raw = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[e]));
        x[2 * e] = f.x;
        x[2 * e + 1] = f.y;
    }
}

template <typename Tin>
__global__ void __launch_bounds__(kPtThreads, 1) gdr_chunk_prep_tc(const __grid_constant__ PrepTcArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kPtBars);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + kPtSlot);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kPtAbort);
    float *Gs = reinterpret_cast<float *>(smem + kPtGs);
    float *bsv = reinterpret_cast<float *>(smem + kPtVec);
    float *gmv = bsv + kPtC, *glv = gmv + kPtD, *g31 = glv + kPtD;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int HV = a.HV;

    // the chunk (as gdr_chunk_prep): dense CTA (b, hv, c), record (b, hv, c);
    // packed CTA (chunk, hv), record (chunk, hv)
    int hv, L;
    size_t tr0, rec_idx;
    if (a.chunks) {
        const int ci = blockIdx.x / HV;
        hv = blockIdx.x % HV;
        const int2 e = a.chunks[ci];
        tr0 = (size_t)e.x;
        L = e.y;
        rec_idx = (size_t)ci * HV + hv;
    } else {
        const int c = blockIdx.x % a.NC;
        const int head_idx = blockIdx.x / a.NC;
        hv = head_idx % HV;
        const int b = head_idx / HV;
        tr0 = (size_t)b * a.T + (size_t)c * kPtC;
        L = min(kPtC, a.T - c * kPtC);
        rec_idx = (size_t)head_idx * a.NC + c;
    }
    const int hk = hv / (HV / a.HK);
    float *rec = a.ws + rec_idx * a.rec_floats;
    unsigned char *rec_b = reinterpret_cast<unsigned char *>(rec);
    // record regions (bytes): Wk, Qt, Kh hi | lo tiles of 32 KB, Wv f32,
    // P hi | lo (16 KB), gam
    constexpr size_t kRegion = (size_t)kPtC * kPtD * 4;
    unsigned char *rec_wk = rec_b, *rec_qt = rec_b + kRegion, *rec_kh = rec_b + 2 * kRegion;
    float *rec_wv = rec + 3 * (size_t)kPtC * kPtD;
    unsigned char *rec_p = rec_b + 4 * kRegion;
    float *rec_gam = rec + 4 * (size_t)kPtC * kPtD + kPtC * kPtC;
    const Tin *qp = static_cast<const Tin *>(a.q), *kp = static_cast<const Tin *>(a.k);
    const Tin *vp = static_cast<const Tin *>(a.v);

    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bars[i], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tslot, 256);

    // this thread's rows of k and q for step 2 (item tid + 256 u: row
    // item % 64, channels 8 (item / 64) ..), loaded before anything waits;
    // the same rows of v go to L2 for the right-hand side built in step 3
    // (rows past L read row L - 1 and are zeroed after the loads, so that
    // every load is issued unconditionally and all are in flight at once)
    float kq[kPtItems][16];
#pragma unroll
    for (int u = 0; u < kPtItems; ++u) {
        const int item = tid + kPtThreads * u;
        const int r = item & 63, i0 = 8 * (item >> 6);
        const int rc = min(r, L - 1);
        const size_t tk = ((tr0 + rc) * a.HK + hk) * kPtD + i0;
        float k8[8], q8[8];
        pt_load8(kp + tk, k8);
        pt_load8(qp + tk, q8);
        prefetch_l2(vp + ((tr0 + rc) * HV + hv) * kPtD + i0);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            kq[u][e] = k8[e];
            kq[u][8 + e] = q8[e];
        }
    }
#pragma unroll
    for (int u = 0; u < kPtItems; ++u) {
        const int r = (tid + kPtThreads * u) & 63;
        if (r >= L) {
#pragma unroll
            for (int e = 0; e < 16; ++e) kq[u][e] = 0.f;
        }
    }

    // ---- 1. prefix sums of the log-decay: threads 0-255, two per key
    // channel i (rows 0-31 and 32-63); the second half adds the first's
    // total after a barrier.  beta on threads 256-319.
    bool in_range = true;
    const int pc = tid & (kPtD - 1), ph = tid >> 7;  // channel, half (tid < 256)
    float gx[32];
    if (tid < 2 * kPtD) {
#pragma unroll
        for (int u = 0; u < 32; ++u) {
            const int r = 32 * ph + u;
            const size_t row = tr0 + min(r, L - 1);
            gx[u] = a.g_scalar ? a.g[row * HV + hv] : a.g[(row * HV + hv) * kPtD + pc];
        }
        float run = 0.f;
#pragma unroll
        for (int u = 0; u < 32; ++u) {
            run += 32 * ph + u < L ? gx[u] : 0.f;  // a zero gate past L keeps G flat
            gx[u] = run;
        }
        if (ph == 0) {
#pragma unroll
            for (int u = 0; u < 32; ++u) Gs[u * kPtLdg + pc] = gx[u];
            g31[pc] = gx[31];
        }
    } else if (tid < 2 * kPtD + kPtC) {
        const int r = tid - 2 * kPtD;
        bsv[r] = r < L ? a.beta[(tr0 + r) * HV + hv] : 0.f;
    }
    __syncthreads();
    if (tid >= kPtD && tid < 2 * kPtD) {
        const float base = g31[pc];
#pragma unroll
        for (int u = 0; u < 32; ++u) Gs[(32 + u) * kPtLdg + pc] = gx[u] + base;
    }
    __syncthreads();
    if (tid < kPtD) {
        const int m = (L - 1) / 2;
        const float gm = Gs[m * kPtLdg + pc], gl = Gs[(L - 1) * kPtLdg + pc];
        gmv[pc] = gm;
        glv[pc] = gl;
        in_range = Gs[pc] - gm <= kPtRange && gm - gl <= kPtRange;
    }
    tc_fence_before_sync();
    const bool fast = __syncthreads_and(in_range) != 0;
    tc_fence_after_sync();
    const uint32_t tmem = *tslot;
    auto wait = [&](int id, uint32_t parity) {
        if (*abort_flag) return;
        if (!mbar_wait_bounded(&bars[id], parity, kPtWaitNs)) {
            *abort_flag = 1;
            if (a.err) atomicExch(a.err, 1);
        }
    };

    // ---- 2. operand tiles and the Qt, Kh records; item = (row r, channels
    // 8o .. 8o + 7), consecutive threads on consecutive rows so that eight
    // of them fill one 128-byte core matrix
#pragma unroll
    for (int u = 0; u < kPtItems; ++u) {
        const int item = tid + kPtThreads * u;
        const int r = item & 63, o = item >> 6, i0 = 8 * o;
        float kk[8], qq[8], G[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            kk[e] = kq[u][e];
            qq[e] = kq[u][8 + e];
        }
        pt_load8(Gs + r * kPtLdg + i0, G);
        const float br = bsv[r];
        float lk[8], lq[8], rr[8], rk[8], qt[8], kh[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float eg = fast_exp2(G[e] * kLog2e);                  // e^G, <= 1
            qt[e] = qq[e] * eg;
            kh[e] = r < L ? kk[e] * fast_exp2((glv[i0 + e] - G[e]) * kLog2e) : 0.f;
            rk[e] = br * kk[e] * eg;
            if (fast) {
                const float d = (G[e] - gmv[i0 + e]) * kLog2e;
                const float up = fast_exp2(d), down = fast_exp2(-d);
                lk[e] = kk[e] * up;
                lq[e] = qq[e] * up;
                rr[e] = kk[e] * down;
            }
        }
        uint4 h, l;
        const uint32_t off = kmajor_off(r, i0, kPtD);
        pt_split8(qt, h, l);
        *reinterpret_cast<uint4 *>(rec_qt + off) = h;
        *reinterpret_cast<uint4 *>(rec_qt + 16384 + off) = l;
        pt_split8(kh, h, l);
        *reinterpret_cast<uint4 *>(rec_kh + off) = h;
        *reinterpret_cast<uint4 *>(rec_kh + 16384 + off) = l;
        pt_split8(rk, h, l);
        *reinterpret_cast<uint4 *>(smem + kPtRk + off) = h;
        *reinterpret_cast<uint4 *>(smem + kPtRk + 16384 + off) = l;
        if (fast) {
            pt_split8(lk, h, l);
            *reinterpret_cast<uint4 *>(smem + kPtAop + off) = h;
            *reinterpret_cast<uint4 *>(smem + kPtAop + 32768 + off) = l;
            const uint32_t offq = kmajor_off(64 + r, i0, kPtD);
            pt_split8(lq, h, l);
            *reinterpret_cast<uint4 *>(smem + kPtAop + offq) = h;
            *reinterpret_cast<uint4 *>(smem + kPtAop + 32768 + offq) = l;
            pt_split8(rr, h, l);
            *reinterpret_cast<uint4 *>(smem + kPtR + off) = h;
            *reinterpret_cast<uint4 *>(smem + kPtR + 16384 + off) = l;
        }
    }
    if (tid < kPtD) rec_gam[tid] = expf(glv[tid]);
    fence_async_smem();
    __syncthreads();

    // ---- 3. the gram [Lk; Lq] R^T (fast chunks) into columns 0-63
    bool issued = false;
    if (fast && tid == 0) {
        tc_fence_after_sync();
        const uint32_t idG = idesc_bf16(128, kPtC, false, false, false);
        const uint32_t sa = smem_u32(smem + kPtAop), sb = smem_u32(smem + kPtR);
        const uint64_t ah = smem_desc(sa, 128, kPtD * 16), al = smem_desc(sa + 32768, 128, kPtD * 16);
        const uint64_t bh = smem_desc(sb, 128, kPtD * 16), bl = smem_desc(sb + 16384, 128, kPtD * 16);
        for (int ks = 0; ks < kPtD / 16; ++ks)
            mma_bf16(tmem, ah + (uint64_t)(16 * ks), bh + (uint64_t)(16 * ks), idG, ks > 0 ? 1u : 0u);
        for (int ks = 0; ks < kPtD / 16; ++ks)
            mma_bf16(tmem, ah + (uint64_t)(16 * ks), bl + (uint64_t)(16 * ks), idG, 1u);
        for (int ks = 0; ks < kPtD / 16; ++ks)
            mma_bf16(tmem, al + (uint64_t)(16 * ks), bh + (uint64_t)(16 * ks), idG, 1u);
        mma_commit(&bars[0]);
        issued = true;
    }
    float *As = reinterpret_cast<float *>(smem + kPtAs);
    float *Tf = reinterpret_cast<float *>(smem + kPtTf);
    if (!fast) {
        // exact pairwise decays: K^T and Q^T staged channel-major, then
        // warp w takes rows r = w, w + 8, ..., lanes the columns s = lane,
        // lane + 32 (s <= r); every exponent G_r - G_s <= 0
        float *KT = reinterpret_cast<float *>(smem + kPtKT);
        float *QT = reinterpret_cast<float *>(smem + kPtQT);
        for (int idx = tid; idx < kPtC * kPtD; idx += kPtThreads) {
            const int r = idx / kPtD, i = idx % kPtD;
            float kv = 0.f, qv = 0.f;
            if (r < L) {
                const size_t tk = ((tr0 + r) * a.HK + hk) * kPtD + i;
                kv = to_f32(kp[tk]);
                qv = to_f32(qp[tk]);
            }
            KT[i * kPtC + r] = kv;
            QT[i * kPtC + r] = qv;
        }
        __syncthreads();
        constexpr int kRowsW = kPtC / kPtWarps;
        float av[kRowsW][2], pv[kRowsW][2];
#pragma unroll
        for (int j = 0; j < kRowsW; ++j) {
            const int r = warp + kPtWarps * j;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int s = lane + 32 * h;
                float sa = 0.f, sp = 0.f;
                if (s <= r && r < L) {
                    for (int i = 0; i < kPtD; ++i) {
                        const float e = fast_exp2((Gs[r * kPtLdg + i] - Gs[s * kPtLdg + i]) * kLog2e);
                        const float ks = KT[i * kPtC + s] * e;
                        sa = fmaf(KT[i * kPtC + r], ks, sa);
                        sp = fmaf(QT[i * kPtC + r], ks, sp);
                    }
                }
                av[j][h] = s < r ? bsv[r] * sa : 0.f;
                pv[j][h] = sp;
            }
        }
        __syncthreads();  // K^T, Q^T read: A and the staged P may overwrite them
#pragma unroll
        for (int j = 0; j < kRowsW; ++j) {
            const int r = warp + kPtWarps * j;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                As[r * kPtLda + lane + 32 * h] = av[j][h];
                Tf[r * kPtLda + lane + 32 * h] = pv[j][h];
            }
        }
        __syncthreads();
        // P into its record: item (row t, columns 8o ..), as in step 2
        for (int item = tid; item < kPtC * 8; item += kPtThreads) {
            const int t = item & 63, o = item >> 6;
            float x[8];
            pt_load8(Tf + t * kPtLda + 8 * o, x);
            uint4 h, l;
            pt_split8(x, h, l);
            const uint32_t off = kmajor_off(t, 8 * o, kPtC);
            *reinterpret_cast<uint4 *>(rec_p + off) = h;
            *reinterpret_cast<uint4 *>(rec_p + 8192 + off) = l;
        }
        __syncthreads();  // G and the staged P read
    }

    // diag(beta) V into the G region (G is no longer read); the four rows'
    // loads in flight together
    {
        float vv[kPtItems][8];
#pragma unroll
        for (int u = 0; u < kPtItems; ++u) {
            const int item = tid + kPtThreads * u;
            const int s = item & 63, j0 = 8 * (item >> 6);
            pt_load8(vp + ((tr0 + min(s, L - 1)) * HV + hv) * kPtD + j0, vv[u]);
        }
#pragma unroll
        for (int u = 0; u < kPtItems; ++u) {
            const int item = tid + kPtThreads * u;
            const int s = item & 63, j0 = 8 * (item >> 6);
            const float bs = bsv[s];  // zero past L
#pragma unroll
            for (int e = 0; e < 8; ++e) vv[u][e] *= bs;
            uint4 h, l;
            pt_split8(vv[u], h, l);
            const uint32_t off = kmajor_off(s, j0, kPtD);
            *reinterpret_cast<uint4 *>(smem + kPtGs + off) = h;
            *reinterpret_cast<uint4 *>(smem + kPtGs + 16384 + off) = l;
        }
    }

    // ---- 4. A and P out of tensor memory: warp w reads lanes 32 (w % 4) ..,
    // columns 16 (w / 4) ..; lanes 0-63 are the rows of A, 64-127 those of P
    if (fast) {
        wait(0, 0);
        if (!*abort_flag) {
            tc_fence_after_sync();
            const int qd = warp & 3, part = warp >> 2;
            float x[16];
            tmem_ld16(tmem + ((uint32_t)(32 * qd) << 16) + 16 * part, x);
            const int lrow = 32 * qd + lane;
            if (lrow < kPtC) {
                const int r = lrow;
                const float br = bsv[r];
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    float4 y;
                    const int s0 = 16 * part + 4 * c4;
                    y.x = (s0 + 0 < r && r < L) ? br * x[4 * c4 + 0] : 0.f;
                    y.y = (s0 + 1 < r && r < L) ? br * x[4 * c4 + 1] : 0.f;
                    y.z = (s0 + 2 < r && r < L) ? br * x[4 * c4 + 2] : 0.f;
                    y.w = (s0 + 3 < r && r < L) ? br * x[4 * c4 + 3] : 0.f;
                    *reinterpret_cast<float4 *>(As + r * kPtLda + s0) = y;
                }
            } else {
                const int t = lrow - kPtC;
#pragma unroll
                for (int oo = 0; oo < 2; ++oo) {
                    float y[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int s = 16 * part + 8 * oo + e;
                        y[e] = (s <= t && t < L) ? x[8 * oo + e] : 0.f;
                    }
                    uint4 h, l;
                    pt_split8(y, h, l);
                    const uint32_t off = kmajor_off(t, 16 * part + 8 * oo, kPtC);
                    *reinterpret_cast<uint4 *>(rec_p + off) = h;
                    *reinterpret_cast<uint4 *>(rec_p + 8192 + off) = l;
                }
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();

    // ---- 5. T = (I + A)^-1 in f32: diagonal blocks (thread (I, j): column j
    // of T_II by forward substitution), then the blocks below them
    if (tid < 64) {
        const int I = tid >> 4, j = tid & 15, b0 = 16 * I;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc = 0.f;
#pragma unroll
            for (int s = 0; s < r; ++s) acc = fmaf(As[(b0 + r) * kPtLda + b0 + s], x[s], acc);
            x[r] = r == j ? 1.f : (r < j ? 0.f : -acc);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) Tf[(b0 + r) * kPtLda + b0 + j] = x[r];
    }
    __syncthreads();
    float *Xs = reinterpret_cast<float *>(smem + kPtX);
#pragma unroll 1
    for (int I = 1; I < 4; ++I) {
        // X_IJ = sum over the blocks K = J .. I-1 of A_IK T_KJ (T is zero
        // above its diagonal); a thread takes a 1 x 4 strip (row r, columns
        // 4 c4 ..) of one block J
        for (int st = tid; st < 64 * I; st += kPtThreads) {
            const int J = st >> 6, r = (st >> 2) & 15, c4 = st & 3;
            const float *arow = As + (16 * I + r) * kPtLda;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int K = J; K < I; ++K) {
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const int uu = 16 * K + t;
                    const float av = arow[uu];
                    const float4 tv = *reinterpret_cast<const float4 *>(Tf + uu * kPtLda + 16 * J + 4 * c4);
                    acc.x = fmaf(av, tv.x, acc.x);
                    acc.y = fmaf(av, tv.y, acc.y);
                    acc.z = fmaf(av, tv.z, acc.z);
                    acc.w = fmaf(av, tv.w, acc.w);
                }
            }
            *reinterpret_cast<float4 *>(Xs + (J << 8) + (r << 4) + 4 * c4) = acc;
        }
        __syncthreads();
        // T_IJ = -T_II X_IJ (T_II unit lower, stored with zeros above its
        // diagonal)
        for (int st = tid; st < 64 * I; st += kPtThreads) {
            const int J = st >> 6, r = (st >> 2) & 15, c4 = st & 3;
            const float *trow = Tf + (16 * I + r) * kPtLda + 16 * I;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) {
                const float tv = trow[rr];
                const float4 xv = *reinterpret_cast<const float4 *>(Xs + (J << 8) + (rr << 4) + 4 * c4);
                acc.x = fmaf(tv, xv.x, acc.x);
                acc.y = fmaf(tv, xv.y, acc.y);
                acc.z = fmaf(tv, xv.z, acc.z);
                acc.w = fmaf(tv, xv.w, acc.w);
            }
            *reinterpret_cast<float4 *>(Tf + (16 * I + r) * kPtLda + 16 * J + 4 * c4) =
                make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
        }
        __syncthreads();
    }
    // T as the A operand: bf16 hi | lo, zero above the diagonal
    for (int item = tid; item < kPtC * 8; item += kPtThreads) {
        const int r = item & 63, o = item >> 6;
        float x[8];
        pt_load8(Tf + r * kPtLda + 8 * o, x);
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (8 * o + e > r) x[e] = 0.f;
        uint4 h, l;
        pt_split8(x, h, l);
        const uint32_t off = kmajor_off(r, 8 * o, kPtC);
        *reinterpret_cast<uint4 *>(smem + kPtT + off) = h;
        *reinterpret_cast<uint4 *>(smem + kPtT + 8192 + off) = l;
    }
    fence_async_smem();
    tc_fence_before_sync();
    __syncthreads();

    // ---- 6. Wk = T RHS_k into columns 0-127, Wv = T RHS_v into 128-255
    if (tid == 0 && !*abort_flag) {
        tc_fence_after_sync();
        const uint32_t idW = idesc_bf16(128, kPtD, false, true, false);
        const uint32_t st = smem_u32(smem + kPtT);
        const uint64_t th = smem_desc(st, 128, kPtC * 16), tl = smem_desc(st + 8192, 128, kPtC * 16);
        for (int part = 0; part < 2; ++part) {
            const uint32_t sr = smem_u32(smem + (part ? kPtGs : kPtRk));
            const uint64_t rh = smem_desc(sr, kPtD * 16, 128), rl = smem_desc(sr + 16384, kPtD * 16, 128);
            const uint32_t d = tmem + 128 * part;
            // 16 rows of the right-hand side per K step: two core matrices along K
            for (int ks = 0; ks < kPtC / 16; ++ks)
                mma_bf16(d, th + (uint64_t)(16 * ks), rh + (uint64_t)(256 * ks), idW, ks > 0 ? 1u : 0u);
            for (int ks = 0; ks < kPtC / 16; ++ks)
                mma_bf16(d, th + (uint64_t)(16 * ks), rl + (uint64_t)(256 * ks), idW, 1u);
            for (int ks = 0; ks < kPtC / 16; ++ks)
                mma_bf16(d, tl + (uint64_t)(16 * ks), rh + (uint64_t)(256 * ks), idW, 1u);
        }
        mma_commit(&bars[1]);
        issued = true;
    }

    // ---- 7. Wk and Wv: the warps of lane quarters 0 and 1 read the 64 rows,
    // warp w columns 64 (w / 4 % 2) .. of Wk (w / 8 = 0) or Wv (w / 8 = 1);
    // Wv is staged in the R region (free once the gram is done)
    float *Wst = reinterpret_cast<float *>(smem + kPtR);
    const int qd = warp & 3, part = warp >> 2;
    if (qd < 2) {
        wait(1, 0);
        if (!*abort_flag) {
            tc_fence_after_sync();
            const int r = 32 * qd + lane;
            const bool is_v = part >= 2;
            const int cb = 64 * (part & 1);
#pragma unroll
            for (int c0 = cb; c0 < cb + 64; c0 += 32) {
                float x[32];
                tmem_ld32(tmem + ((uint32_t)(32 * qd) << 16) + (is_v ? 128 : 0) + c0, x);
                if (!is_v) {
#pragma unroll
                    for (int oo = 0; oo < 4; ++oo) {
                        float y[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) y[e] = x[8 * oo + e];
                        uint4 h, l;
                        pt_split8(y, h, l);
                        const uint32_t off = kmajor_off(r, c0 + 8 * oo, kPtD);
                        *reinterpret_cast<uint4 *>(rec_wk + off) = h;
                        *reinterpret_cast<uint4 *>(rec_wk + 16384 + off) = l;
                    }
                } else {
                    // row r into the staging tile, 16-byte chunks XORed with
                    // r % 8 so that eight rows at once hit distinct banks
#pragma unroll
                    for (int c4 = 0; c4 < 8; ++c4) {
                        const int ch = ((c0 >> 2) + c4) ^ (r & 7);
                        *reinterpret_cast<float4 *>(Wst + r * kPtD + 4 * ch) =
                            make_float4(x[4 * c4], x[4 * c4 + 1], x[4 * c4 + 2], x[4 * c4 + 3]);
                    }
                }
            }
        }
    }
    __syncthreads();
    // Wv from the staging tile to its record, each warp two full rows per store
    if (!*abort_flag) {
#pragma unroll
        for (int u = 0; u < 64 * 32 / kPtThreads; ++u) {
            const int idx = tid + kPtThreads * u;  // float4 index in [64][32]
            const int r = idx >> 5, ch = idx & 31;
            *reinterpret_cast<float4 *>(rec_wv + r * kPtD + 4 * ch) =
                *reinterpret_cast<const float4 *>(Wst + r * kPtD + 4 * (ch ^ (r & 7)));
        }
    }

    // every MMA issued is done before the tensor memory is released
    if (issued && *abort_flag) {
        mma_commit(&bars[2]);
        mbar_wait_bounded(&bars[2], 0, kPtWaitNs);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

}  // namespace

// float32 q/k/v (bf16 at this shape takes the fused tensor-core prefill)
bool prep_tc_supported(const Problem &p) {
    return !p.bf16 && p.dk == kPtD && p.dv == kPtD && p.chunk == kPtC;
}

cudaError_t launch_chunk_prep_tc(const Problem &p, float *records, size_t rec_floats,
                                 const int2 *chunks, int nchunks, cudaStream_t stream) {
    if (!prep_tc_supported(p)) return cudaErrorInvalidValue;
    int *err = nullptr;
    cudaError_t e = device_error_word(&err);
    if (e != cudaSuccess) return e;
    PrepTcArgs a;
    a.q = p.q; a.k = p.k; a.v = p.v; a.g = p.g; a.beta = p.beta; a.ws = records;
    a.chunks = chunks; a.err = err;
    a.T = p.T; a.HK = p.HK; a.HV = p.HV; a.NC = (p.T + kPtC - 1) / kPtC; a.g_scalar = p.g_scalar;
    a.rec_floats = rec_floats;
    const long long ctas = chunks ? (long long)nchunks * p.HV : (long long)p.B * p.HV * a.NC;
    if (ctas == 0) return cudaSuccess;
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if ((e = cudaFuncSetAttribute(gdr_chunk_prep_tc<float>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPtSmem)) !=
        cudaSuccess)
        return e;
    trace_begin(kKernChunkPrepTc, stream);
    gdr_chunk_prep_tc<float><<<(unsigned)ctas, kPtThreads, kPtSmem, stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    trace_end(kKernChunkPrepTc, stream);
    return cudaSuccess;
}

}  // namespace gdr
