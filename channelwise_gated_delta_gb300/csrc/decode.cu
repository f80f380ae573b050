// decode.cu -- single-token (T == 1) channelwise gated delta rule step.
//
// Page "Reorder channelwise gated delta rule chunked hot loops for
// autovectorization" (pytorch/executorch PR #21021), first commit summary:
// the four state traversals of a token (decay, predict, update, output) are
// folded into two -- a first pass that predicts with the decay folded in and
// a second that applies decay plus the rank-one update while accumulating the
// output.  On the GPU the state tile is held in registers between the two
// passes, so the float32 state is read from HBM exactly once and written
// exactly once; that traffic (8 bytes per state element) is the whole cost.
//
// Work split: one CTA per (batch, value head, 32-column tile of dv), 2*DK
// threads.  Thread (cq = tid % 8, rg = tid / 8) owns columns
// [32*tile + 4*cq, +4) of rows rg + (DK/4)*m, m = 0..3, loaded and stored as
// 16-byte vectors.  A warp therefore touches four 128-byte row segments per
// access.  Column sums over the DK rows (vhat = S^T k and o = S^T q) are
// reduced with warp shuffles across the four row groups of a warp, then
// across warps through shared memory.
#include "common.cuh"
#include "sm100_ptx.cuh"

namespace gdr {
namespace {

constexpr int kDecodeBV = 32;  // value columns per CTA

__device__ __forceinline__ float4 f4_fma(float a, float4 x, float4 acc) {
    acc.x = fmaf(a, x.x, acc.x);
    acc.y = fmaf(a, x.y, acc.y);
    acc.z = fmaf(a, x.z, acc.z);
    acc.w = fmaf(a, x.w, acc.w);
    return acc;
}

// Sum over the lanes of a warp that share (lane % 8), i.e. over the warp's
// four row groups; every lane ends with the sum for its own column quad.
__device__ __forceinline__ float4 reduce_row_groups(float4 a) {
#pragma unroll
    for (int off = 8; off < 32; off <<= 1) {
        a.x += __shfl_xor_sync(0xffffffffu, a.x, off);
        a.y += __shfl_xor_sync(0xffffffffu, a.y, off);
        a.z += __shfl_xor_sync(0xffffffffu, a.z, off);
        a.w += __shfl_xor_sync(0xffffffffu, a.w, off);
    }
    return a;
}

template <int NW>
__device__ __forceinline__ float4 block_column_sum(float4 part, float (*red)[kDecodeBV], int warp,
                                                   int lane, int cq) {
    part = reduce_row_groups(part);
    if (lane < 8) {
        red[warp][4 * cq + 0] = part.x;
        red[warp][4 * cq + 1] = part.y;
        red[warp][4 * cq + 2] = part.z;
        red[warp][4 * cq + 3] = part.w;
    }
    __syncthreads();
    float4 tot = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        tot.x += red[w][4 * cq + 0];
        tot.y += red[w][4 * cq + 1];
        tot.z += red[w][4 * cq + 2];
        tot.w += red[w][4 * cq + 3];
    }
    return tot;
}

// GS: a scalar gate, g[head] (one log-decay per token and value head).
template <typename Tin, int DK, bool HAS_H0, bool STORE_HT, bool ROWS, bool GS>
__global__ void __launch_bounds__(2 * DK)
    gdr_decode_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                      const Tin *__restrict__ v, const float *__restrict__ g,
                      const float *__restrict__ beta, const float *h0, Tin *__restrict__ out,
                      float *ht, const int2 *__restrict__ rows, int HK, int HV, int dv) {
    constexpr int NT = 2 * DK;
    constexpr int NW = NT / 32;
    constexpr int RG = DK / 4;  // row groups; each thread holds 4 rows
    __shared__ float red1[NW][kDecodeBV];
    __shared__ float red2[NW][kDecodeBV];

    const int ntile = dv / kDecodeBV;
    const int tile = blockIdx.x % ntile;
    const int head_idx = blockIdx.x / ntile;  // b * HV + hv
    const int hv = head_idx % HV;
    const int b = head_idx / HV;
    const int hk = hv / (HV / HK);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cq = tid & 7, rg = tid >> 3;
    const int col = tile * kDecodeBV + 4 * cq;
    // token row and state slot of this batch element: both b, or for one
    // token of a packed variable-length batch, taken from `rows`
    int trow = b;
    size_t head = (size_t)head_idx;  // token-major: q/k/v/g/beta/out
    size_t shead = head;             // state-major: h0/ht
    if (ROWS) {
        const int2 r = rows[b];
        trow = r.x;
        head = (size_t)r.x * HV + hv;
        shead = (size_t)r.y * HV + hv;
    }

    const Tin *kp = k + ((size_t)trow * HK + hk) * DK;
    const Tin *qp = q + ((size_t)trow * HK + hk) * DK;
    const float *gp = g + head * (GS ? 1 : DK);
    const float bt = beta[head];
    const float4 vv = load4(v + head * dv + col);

    // Pass 1: load the tile once, decay it, and form the partial prediction.
    float4 s[4];
    float kr[4], qr[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const int r = rg + RG * m;
        if (HAS_H0) {
            s[m] = ldg_stream4(h0 + (shead * DK + r) * dv + col);
        } else {
            s[m] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        kr[m] = to_f32(kp[r]);
        qr[m] = to_f32(qp[r]);
        const float gamma = expf(gp[GS ? 0 : r]);
        s[m].x *= gamma;
        s[m].y *= gamma;
        s[m].z *= gamma;
        s[m].w *= gamma;
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < 4; ++m) acc = f4_fma(kr[m], s[m], acc);
    const float4 vhat = block_column_sum<NW>(acc, red1, warp, lane, cq);

    // Pass 2: rank-one update in registers, output partials, single store.
    float4 u;
    u.x = bt * (vv.x - vhat.x);
    u.y = bt * (vv.y - vhat.y);
    u.z = bt * (vv.z - vhat.z);
    u.w = bt * (vv.w - vhat.w);
    float4 oacc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        s[m] = f4_fma(kr[m], u, s[m]);
        oacc = f4_fma(qr[m], s[m], oacc);
        if (STORE_HT) stg_stream4(ht + (shead * DK + rg + RG * m) * dv + col, s[m]);
    }
    const float4 o = block_column_sum<NW>(oacc, red2, warp, lane, cq);
    if (tid < 8) store4(out + head * dv + col, o);
}

// ---- dk = dv = 128: persistent, the 64 KB state of a head moved by bulk copies.
//
// One CTA per SM (256 threads) walks heads blockIdx.x, + gridDim.x, ...
// through three shared-memory buffers: the state of head n + 2 and its k, q,
// v rows are loading (one cp.async.bulk each, counted on the buffer's
// mbarrier) while head n computes and the bulk store of head n - 1 drains.
// Thread (j, h) owns column j and rows 64 h .. 64 h + 63: it keeps its 64
// decayed entries in registers through the prediction, updates them, and
// writes them back to the buffer for the output sum and the store.
constexpr int kBulkD = 128;
constexpr int kBulkThreads = 256;
constexpr int kBulkBufs = 3;
constexpr uint32_t kBulkStateBytes = kBulkD * kBulkD * 4;
constexpr uint32_t kBulkVecBytes = 4 * kBulkD * 4;   // k, q, v, g rows (room for f32)
constexpr uint32_t kBulkBufBytes = kBulkStateBytes + kBulkVecBytes;
constexpr uint64_t kBulkWaitNs = 2000000000ull;  // 2 s

template <typename Tin, bool HAS_H0, bool STORE_HT, bool ROWS, bool GS>
__global__ void __launch_bounds__(kBulkThreads, 1)
    gdr_decode_bulk_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                           const Tin *__restrict__ v, const float *__restrict__ g,
                           const float *__restrict__ beta, const float *h0,
                           Tin *__restrict__ out, float *ht, const int2 *__restrict__ rows, int HK,
                           int HV, int nheads, int *dev_error) {
    extern __shared__ float4 smem_f4[];
    unsigned char *base = reinterpret_cast<unsigned char *>(smem_f4);
    float *red = reinterpret_cast<float *>(base + kBulkBufs * kBulkBufBytes);  // [2][128]
    float *gam = red + 2 * kBulkD;                                               // exp(g) [128]
    float *kf = gam + kBulkD;                                                    // k as f32 [128]
    float *qf = kf + kBulkD;                                                     // q as f32 [128]
    uint64_t *bars = reinterpret_cast<uint64_t *>(qf + kBulkD);                 // [kBulkBufs]
    const int tid = threadIdx.x, j = tid & (kBulkD - 1), half = tid >> 7;
    constexpr uint32_t es = sizeof(Tin);

    // token row, state slot and key head of the CTA's n-th head
    auto head_of = [&](int n, size_t &head, size_t &shead, size_t &krow) {
        const int head_idx = blockIdx.x + n * gridDim.x;
        const int hv = head_idx % HV, b = head_idx / HV;
        int trow = b;
        head = (size_t)head_idx;
        shead = head;
        if (ROWS) {
            const int2 r = rows[b];
            trow = r.x;
            head = (size_t)r.x * HV + hv;
            shead = (size_t)r.y * HV + hv;
        }
        krow = (size_t)trow * HK + hv / (HV / HK);
    };
    auto buf = [&](int n) { return base + (n % kBulkBufs) * kBulkBufBytes; };
    // thread 0: the loads of the CTA's n-th head into its buffer
    auto issue = [&](int n) {
        size_t head, shead, krow;
        head_of(n, head, shead, krow);
        unsigned char *bp = buf(n);
        uint64_t *bar = bars + n % kBulkBufs;
        const uint32_t bytes = (HAS_H0 ? kBulkStateBytes : 0u) + 3 * kBulkD * es +
                               (GS ? 0u : kBulkD * 4u);
        sm100::mbar_arrive_expect_tx(bar, bytes);
        if (HAS_H0) sm100::bulk_load_1d(bp, h0 + shead * kBulkD * kBulkD, kBulkStateBytes, bar);
        unsigned char *vp = bp + kBulkStateBytes;
        sm100::bulk_load_1d(vp, k + krow * kBulkD, kBulkD * es, bar);
        sm100::bulk_load_1d(vp + 512, q + krow * kBulkD, kBulkD * es, bar);
        sm100::bulk_load_1d(vp + 1024, v + head * kBulkD, kBulkD * es, bar);
        if (!GS) sm100::bulk_load_1d(vp + 1536, g + head * kBulkD, kBulkD * 4u, bar);
    };
    const int my = blockIdx.x < nheads ? (nheads - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    if (tid == 0) {
        for (int i = 0; i < kBulkBufs; ++i) sm100::mbar_init(bars + i, 1);
        sm100::fence_mbar_init();
        for (int n = 0; n < kBulkBufs - 1 && n < my; ++n) issue(n);
    }
    __syncthreads();

    // beta (and a scalar gate's g) of the next head are read one head ahead,
    // so that their latency hides behind a head's work
    float bt_next = 0.f, gs_next = 0.f;
    if (my > 0) {
        size_t head, shead, krow;
        head_of(0, head, shead, krow);
        bt_next = beta[head];
        if (GS) gs_next = g[head];
    }
    int n = 0;
    for (; n < my; ++n) {
        if (tid == 0 && n + kBulkBufs - 1 < my) {
            // the buffer of head n + 2 last held head n - 1: its store must
            // have read it
            sm100::bulk_wait_read_all();
            issue(n + kBulkBufs - 1);
        }
        size_t head, shead, krow;
        head_of(n, head, shead, krow);
        const float bt = bt_next, gs = gs_next;
        if (n + 1 < my) {
            size_t h1, s1, k1;
            head_of(n + 1, h1, s1, k1);
            bt_next = beta[h1];
            if (GS) gs_next = g[h1];
        }
        const bool ok = __syncthreads_and(
            sm100::mbar_wait_bounded(bars + n % kBulkBufs, (uint32_t)((n / kBulkBufs) & 1),
                                     kBulkWaitNs)) != 0;
        if (!ok) {
            if (tid == 0) atomicOr(dev_error, 1);
            break;
        }
        float *S = reinterpret_cast<float *>(buf(n));
        const Tin *kv = reinterpret_cast<const Tin *>(buf(n) + kBulkStateBytes);
        const Tin *qv = reinterpret_cast<const Tin *>(buf(n) + kBulkStateBytes + 512);
        const Tin *vv = reinterpret_cast<const Tin *>(buf(n) + kBulkStateBytes + 1024);
        // per row, once: the decay exp(g) and k, q as f32
        if (tid < kBulkD) {
            gam[tid] = expf(GS ? gs
                               : reinterpret_cast<const float *>(buf(n) + kBulkStateBytes + 1536)[tid]);
            kf[tid] = to_f32(kv[tid]);
            qf[tid] = to_f32(qv[tid]);
        }
        __syncthreads();
        // pass 1: decayed entries kept in registers, partial prediction
        float s[64];
        float acc = 0.f;
#pragma unroll
        for (int r = 0; r < 64; ++r) {
            const int i = 64 * half + r;
            const float x = HAS_H0 ? S[i * kBulkD + j] * gam[i] : 0.f;
            s[r] = x;
            acc = fmaf(kf[i], x, acc);
        }
        red[half * kBulkD + j] = acc;
        __syncthreads();
        const float u = bt * (to_f32(vv[j]) - (red[j] + red[kBulkD + j]));
        __syncthreads();  // both halves have read red before it is reused
        // pass 2: rank-one update, output partials, the tile back in the buffer
        float o = 0.f;
#pragma unroll
        for (int r = 0; r < 64; ++r) {
            const int i = 64 * half + r;
            const float x = fmaf(kf[i], u, s[r]);
            o = fmaf(qf[i], x, o);
            if (STORE_HT) S[i * kBulkD + j] = x;
        }
        red[half * kBulkD + j] = o;
        if (STORE_HT) sm100::fence_async_smem();  // generic writes, before the bulk store reads
        __syncthreads();
        if (tid < kBulkD) out[head * kBulkD + tid] = from_f32<Tin>(red[tid] + red[kBulkD + tid]);
        if (STORE_HT && tid == 0) {
            sm100::bulk_store_1d(ht + shead * kBulkD * kBulkD, S, kBulkStateBytes);
            sm100::bulk_commit_group();
        }
        __syncthreads();  // red is free again
    }
    if (tid == 0) {
        sm100::bulk_wait_all();
        // after a timeout at head n, never leave with loads in flight into
        // this CTA: heads n .. n + 2 may have been issued
        for (int m = n; m < my && m < n + kBulkBufs; ++m)
            sm100::mbar_wait_bounded(bars + m % kBulkBufs, (uint32_t)((m / kBulkBufs) & 1),
                                     kBulkWaitNs);
    }
}

template <typename Tin, bool ROWS, bool GS>
cudaError_t launch_decode_bulk(const Problem &p, const int2 *rows, cudaStream_t stream) {
    const long long nheads = (long long)p.B * p.HV;
    if (nheads > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    int *err = nullptr;
    cudaError_t e = device_error_word(&err);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    const int grid = (int)(nheads < sms ? nheads : sms);
    const size_t smem = kBulkBufs * kBulkBufBytes + 5 * kBulkD * sizeof(float) + 8 * kBulkBufs;
    const Tin *q = static_cast<const Tin *>(p.q), *k = static_cast<const Tin *>(p.k);
    const Tin *v = static_cast<const Tin *>(p.v);
    Tin *out = static_cast<Tin *>(p.out);
    auto run = [&](auto kernel) -> cudaError_t {
        cudaError_t err2 = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                (int)smem);
        if (err2 != cudaSuccess) return err2;
        trace_begin(kKernDecode, stream);
        kernel<<<grid, kBulkThreads, smem, stream>>>(q, k, v, p.g, p.beta, p.h0, out, p.ht, rows,
                                                     p.HK, p.HV, (int)nheads, err);
        trace_end(kKernDecode, stream);
        return cudaGetLastError();
    };
    if (p.h0 && p.ht) return run(gdr_decode_bulk_kernel<Tin, true, true, ROWS, GS>);
    if (p.h0) return run(gdr_decode_bulk_kernel<Tin, true, false, ROWS, GS>);
    if (p.ht) return run(gdr_decode_bulk_kernel<Tin, false, true, ROWS, GS>);
    return run(gdr_decode_bulk_kernel<Tin, false, false, ROWS, GS>);
}

template <typename Tin, int DK, bool ROWS, bool GS>
cudaError_t launch_decode_t(const Problem &p, const int2 *rows, cudaStream_t stream) {
    const long long blocks = (long long)p.B * p.HV * (p.dv / kDecodeBV);
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    dim3 grid((unsigned)blocks), block(2 * DK);
    const Tin *q = static_cast<const Tin *>(p.q), *k = static_cast<const Tin *>(p.k);
    const Tin *v = static_cast<const Tin *>(p.v);
    Tin *out = static_cast<Tin *>(p.out);
    trace_begin(kKernDecode, stream);
    if (p.h0 && p.ht)
        gdr_decode_kernel<Tin, DK, true, true, ROWS, GS><<<grid, block, 0, stream>>>(
            q, k, v, p.g, p.beta, p.h0, out, p.ht, rows, p.HK, p.HV, p.dv);
    else if (p.h0)
        gdr_decode_kernel<Tin, DK, true, false, ROWS, GS><<<grid, block, 0, stream>>>(
            q, k, v, p.g, p.beta, p.h0, out, p.ht, rows, p.HK, p.HV, p.dv);
    else if (p.ht)
        gdr_decode_kernel<Tin, DK, false, true, ROWS, GS><<<grid, block, 0, stream>>>(
            q, k, v, p.g, p.beta, p.h0, out, p.ht, rows, p.HK, p.HV, p.dv);
    else
        gdr_decode_kernel<Tin, DK, false, false, ROWS, GS><<<grid, block, 0, stream>>>(
            q, k, v, p.g, p.beta, p.h0, out, p.ht, rows, p.HK, p.HV, p.dv);
    trace_end(kKernDecode, stream);
    return cudaGetLastError();
}

template <typename Tin, bool ROWS, bool GS>
cudaError_t launch_decode_d(const Problem &p, const int2 *rows, cudaStream_t stream) {
    if (p.dk == kBulkD && p.dv == kBulkD) return launch_decode_bulk<Tin, ROWS, GS>(p, rows, stream);
    switch (p.dk) {
        case 32: return launch_decode_t<Tin, 32, ROWS, GS>(p, rows, stream);
        case 64: return launch_decode_t<Tin, 64, ROWS, GS>(p, rows, stream);
        case 128: return launch_decode_t<Tin, 128, ROWS, GS>(p, rows, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <typename Tin, bool ROWS>
cudaError_t launch_decode_dt(const Problem &p, const int2 *rows, cudaStream_t stream) {
    return p.g_scalar ? launch_decode_d<Tin, ROWS, true>(p, rows, stream)
                      : launch_decode_d<Tin, ROWS, false>(p, rows, stream);
}

}  // namespace

cudaError_t launch_decode(const Problem &p, cudaStream_t stream) {
    return p.bf16 ? launch_decode_dt<__nv_bfloat16, false>(p, nullptr, stream)
                  : launch_decode_dt<float, false>(p, nullptr, stream);
}

cudaError_t launch_decode_rows(const Problem &p, const int2 *rows, cudaStream_t stream) {
    return p.bf16 ? launch_decode_dt<__nv_bfloat16, true>(p, rows, stream)
                  : launch_decode_dt<float, true>(p, rows, stream);
}

}  // namespace gdr
