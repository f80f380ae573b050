// tma_host.h -- host-side encoding of TMA tensor maps over the library's
// [B][T][H][128] token tensors, shared by the tensor-core kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

namespace gdr {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point, looked up once.
inline EncodeTiledFn tma_encode_fn(cudaError_t *err) {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    static cudaError_t status = cudaSuccess;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        status = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                  cudaEnableDefault, &q);
        if (status == cudaSuccess && q != cudaDriverEntryPointSuccess) status = cudaErrorNotSupported;
        fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    *err = status;
    return fn;
}

// [B][T][H][128] tensor of `esize`-byte elements; boxes of `box_inner`
// elements x `box_rows` tokens of one head, zero fill outside the tensor.
inline bool tma_encode_rows(EncodeTiledFn fn, CUtensorMap *m, const void *base,
                            CUtensorMapDataType dt, int esize, int B, int T, int H, int box_inner,
                            CUtensorMapSwizzle swizzle, int box_rows) {
    const cuuint64_t dims[4] = {128, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)128 * esize, (cuuint64_t)H * 128 * esize,
                                   (cuuint64_t)T * H * 128 * esize};
    const cuuint32_t box[4] = {(cuuint32_t)box_inner, 1, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, dt, 4, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace gdr
