// tq_tmap.cu -- tensor-map encoding through the driver entry point (resolved
// once through the runtime, so libtq needs no link-time libcuda dependency).
#include <mutex>

#include "tq_tmap.h"

namespace tq {

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn(cudaError_t *err) {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    static cudaError_t status = cudaSuccess;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        status = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                  cudaEnableDefault, &q);
        if (status == cudaSuccess && (q != cudaDriverEntryPointSuccess || p == nullptr))
            status = cudaErrorSymbolNotFound;
        fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    *err = status;
    return fn;
}

}  // namespace

cudaError_t make_tmap_2d(CUtensorMap *out, CUtensorMapDataType dtype, const void *base,
                         uint64_t inner, uint64_t rows, uint64_t row_stride_bytes,
                         uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
    cudaError_t e = cudaSuccess;
    EncodeTiledFn fn = encode_fn(&e);
    if (e != cudaSuccess) return e;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_stride_bytes)};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t elem_strides[2] = {1, 1};
    const CUresult r = fn(out, dtype, 2, const_cast<void *>(base), dims, strides, box, elem_strides,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_codes_tmap_3d(CUtensorMap *out, const void *base, uint64_t row_bytes, uint64_t rows) {
    cudaError_t e = cudaSuccess;
    EncodeTiledFn fn = encode_fn(&e);
    if (e != cudaSuccess) return e;
    const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(row_bytes / 128), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(row_bytes)};
    const cuuint32_t box[3] = {128, 2, 16};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    const CUresult r = fn(out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box,
                          elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace tq
