// tmap.cu -- host-side encoding of TMA tensor maps.  The driver entry point
// cuTensorMapEncodeTiled is fetched through the runtime, so the library needs no
// link-time dependency on libcuda.
#include <cuda.h>
#include <cuda_runtime.h>
#include <mutex>

#include "launch.h"

namespace ssm {

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::mutex g_mu;
EncodeTiledFn g_encode = nullptr;

cudaError_t encoder(EncodeTiledFn* out) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_encode == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || fn == nullptr) return cudaErrorNotSupported;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    *out = g_encode;
    return cudaSuccess;
}

}  // namespace

// 2-D row-major tensor [rows][inner] of 2- or 4-byte elements, 128-byte swizzled boxes of
// box_inner x box_rows elements, zero fill outside the tensor.
cudaError_t encode_tmap_2d(CUtensorMap* map, const void* base, int elem_bytes,
                           unsigned long long inner, unsigned long long rows, unsigned box_inner,
                           unsigned box_rows, bool swizzle128) {
    EncodeTiledFn fn = nullptr;
    cudaError_t e = encoder(&fn);
    if (e != cudaSuccess) return e;
    const CUtensorMapDataType dt =
        elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner * static_cast<uint64_t>(elem_bytes)};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Row-major tensor of `rank` dimensions (dims[0] innermost), contiguous strides.
cudaError_t encode_tmap_nd(CUtensorMap* map, const void* base, int elem_bytes, int rank,
                           const unsigned long long* dims, const unsigned* box, bool swizzle128) {
    EncodeTiledFn fn = nullptr;
    cudaError_t e = encoder(&fn);
    if (e != cudaSuccess) return e;
    if (rank < 1 || rank > 5) return cudaErrorInvalidValue;
    const CUtensorMapDataType dt =
        elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    cuuint64_t gd[5], gs[4];
    cuuint32_t bx[5], es[5];
    unsigned long long stride = static_cast<unsigned long long>(elem_bytes);
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i > 0) gs[i - 1] = stride;
        stride *= dims[i];
    }
    CUresult r = fn(map, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(base), gd, gs, bx, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace ssm
