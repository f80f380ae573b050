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
