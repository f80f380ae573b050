// umma_layouts.cu -- test-only diagnostic library (libgdr_diag.so, not part
// of the product library): one tensor-core GEMM through the shared-memory
// operand layouts, descriptors, MMA issue and TMEM read-back that the
// tensor-core kernels use, so that a layout or descriptor fault can be told
// apart from an algebra fault.  D[128 x N] = A[128 x 64] * B[N x 64]^T, bf16
// in, f32 out.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "sm100_ptx.cuh"

namespace gdr {
namespace {

using namespace sm100;

constexpr int kM = 128, kK = 64;

__global__ void __launch_bounds__(128, 1)
    gdr_selftest_umma_kernel(const __nv_bfloat16 *__restrict__ A, const __nv_bfloat16 *__restrict__ B,
                             float *__restrict__ D, int N, int a_mn, int b_mn, int *dev_error) {
    __shared__ __align__(1024) unsigned char sa[kM * kK * 2];
    __shared__ __align__(1024) unsigned char sb[128 * kK * 2];
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t slot;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (warp == 0) tmem_alloc(&slot, 256);
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    // Layout modes: 0 = K-major (row m or n), 1 = MN-major, 2 = a K-major tile
    // of the transpose (rows k, K extent M or N) read back through an MN-major
    // descriptor with LBO and SBO swapped in role, 3 = MN-major with the
    // 128-byte swizzle, 5 = K-major with the 128-byte swizzle (rows of 64
    // elements, 8-row atoms).
    for (int idx = tid; idx < kM * kK; idx += 128) {
        const int m = idx / kK, k = idx % kK;
        const uint32_t off = a_mn == 5   ? sw128_kmajor_off(m, k, kM)
                             : a_mn == 3 ? sw128_mnmajor_off(k, m, kK)
                             : a_mn == 2 ? kmajor_off(k, m, kM)
                             : a_mn == 1 ? mnmajor_off(k, m, kK)
                                         : kmajor_off(m, k, kK);
        *reinterpret_cast<__nv_bfloat16 *>(sa + off) = A[idx];
    }
    for (int idx = tid; idx < N * kK; idx += 128) {
        const int n = idx / kK, k = idx % kK;
        const uint32_t off = b_mn == 5   ? sw128_kmajor_off(n, k, N)
                             : b_mn == 3 ? sw128_mnmajor_off(k, n, kK)
                             : b_mn == 2 ? kmajor_off(k, n, N)
                             : b_mn == 1 ? mnmajor_off(k, n, kK)
                                         : kmajor_off(n, k, kK);
        *reinterpret_cast<__nv_bfloat16 *>(sb + off) = B[idx];
    }
    fence_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = slot;
    if (a_mn == 4) {
        // A in tensor memory: row m in lane m, (A[m][2c], A[m][2c+1]) packed in column 128 + c
        const int m = 32 * warp + lane;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t w[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                __nv_bfloat162 pr;
                pr.x = A[m * kK + 32 * h + 2 * c];
                pr.y = A[m * kK + 32 * h + 2 * c + 1];
                w[c] = *reinterpret_cast<uint32_t *>(&pr);
            }
            tmem_st16(tmem + ((uint32_t)(32 * warp) << 16) + 128 + 16 * h, w);
        }
        tmem_st_wait();
        tc_fence_before_sync();
        __syncthreads();
        tc_fence_after_sync();
    }
    if (tid == 0) {
        const bool a_t = a_mn != 0 && a_mn != 5, b_t = b_mn != 0 && b_mn != 5;  // MN-major
        const uint32_t idesc = idesc_bf16(kM, N, a_t, b_t, false);
        // K-direction / MN-direction core-matrix strides of each operand
        const uint32_t a_lbo = a_mn == 2 ? kM * 16 : 128, a_sbo = a_mn == 2 ? 128 : kK * 16;
        const uint32_t b_lbo = b_mn == 2 ? N * 16 : 128, b_sbo = b_mn == 2 ? 128 : kK * 16;
        for (int ks = 0; ks < kK / 16 && a_mn == 4; ++ks) {
            const uint64_t bd =
                b_mn == 5   ? smem_desc_sw128(smem_u32(sb) + ks * 32, 16, 1024)
                : b_mn == 3 ? smem_desc_sw128(smem_u32(sb) + ks * 2048, kK * 128, 1024)
                            : smem_desc(smem_u32(sb) + ks * 2 * b_lbo, b_lbo, b_sbo);
            mma_bf16_ts(tmem, tmem + 128 + 8 * ks, bd, idesc_bf16(kM, N, false, b_t, false),
                        ks > 0 ? 1u : 0u);
        }
        for (int ks = 0; ks < kK / 16 && a_mn != 4; ++ks) {
            // swizzled MN-major: 64-element blocks of kK rows (LBO), 8-row atoms (SBO)
            // K-major swizzled: each K step of 16 elements advances the start
            // address by 32 bytes inside the 128-byte row (the swizzle is applied
            // to the absolute address); LBO is not used
            const uint64_t ad =
                a_mn == 5   ? smem_desc_sw128(smem_u32(sa) + ks * 32, 16, 1024)
                : a_mn == 3 ? smem_desc_sw128(smem_u32(sa) + ks * 2048, kK * 128, 1024)
                            : smem_desc(smem_u32(sa) + ks * 2 * a_lbo, a_lbo, a_sbo);
            const uint64_t bd =
                b_mn == 5   ? smem_desc_sw128(smem_u32(sb) + ks * 32, 16, 1024)
                : b_mn == 3 ? smem_desc_sw128(smem_u32(sb) + ks * 2048, kK * 128, 1024)
                            : smem_desc(smem_u32(sb) + ks * 2 * b_lbo, b_lbo, b_sbo);
            mma_bf16(tmem, ad, bd, idesc, ks > 0 ? 1u : 0u);
        }
        mma_commit(&bar);
    }
    const bool ok = mbar_wait_bounded(&bar, 0, 2000000000ull);
    const bool all_ok = __syncthreads_and(ok ? 1 : 0) != 0;
    tc_fence_after_sync();
    if (all_ok) {
        const int row = 32 * warp + lane;
        for (int c0 = 0; c0 < N; c0 += 32) {
            float d[32];
            tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + c0, d);
#pragma unroll
            for (int u = 0; u < 32; ++u) D[row * N + c0 + u] = d[u];
        }
    } else if (tid == 0) {
        atomicOr(dev_error, 1);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 256);
    }
}

}  // namespace
}  // namespace gdr

// D[128 x N] = A[128 x 64] * B[N x 64]^T (row-major bf16 in, row-major f32
// out, device pointers), N in {64, 128}; a_mode (0-5) and b_mode (0-3, 5)
// select the operand layouts listed in the kernel, a_mode 4 puts A in tensor
// memory.  `err` is a device int that a timed-out wait sets to 1.  Returns 0,
// or -1 for bad arguments, or the cudaError_t of the launch.
extern "C" __attribute__((visibility("default"))) int gdr_diag_umma(int a_mode, int b_mode, int N,
                                                                   const void *A, const void *B,
                                                                   float *D, int *err,
                                                                   void *stream) {
    if (!A || !B || !D || !err) return -1;
    if (N != 64 && N != 128) return -1;
    if (a_mode < 0 || a_mode > 5 || b_mode < 0 || b_mode > 5 || b_mode == 4) return -1;
    gdr::gdr_selftest_umma_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const __nv_bfloat16 *>(A), static_cast<const __nv_bfloat16 *>(B), D, N,
        a_mode, b_mode, err);
    return (int)cudaGetLastError();
}

