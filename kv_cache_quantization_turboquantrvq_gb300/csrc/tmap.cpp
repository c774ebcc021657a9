// tmap.cpp - host-side encoding of TMA tensor maps (the descriptors that
// cp.async.bulk.tensor reads).  The driver's encoder is looked up once
// through the runtime, so the library links against the CUDA runtime only.
#include <cuda.h>
#include <cuda_runtime_api.h>

#include <mutex>

#include "launch.h"

namespace vq {

namespace {

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                 CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                 CUtensorMapFloatOOBfill);

EncodeTiled encoder()
{
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    });
    return fn;
}

}  // namespace

bool encode_tmap_f16(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                     const uint64_t *strides, const uint32_t *box, bool swizzle128, bool promote256)
{
    EncodeTiled fn = encoder();
    if (fn == nullptr || rank < 1 || rank > 5) return false;
    cuuint64_t gd[5], gs[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) gs[i] = strides[i];
    }
    const CUresult r =
        fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (cuuint32_t)rank, const_cast<void *>(base), gd, gs, bx, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
           promote256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_tmap_words(CUtensorMap *map, const void *base, uint64_t rows, uint32_t words, uint32_t box_rows,
                       int swizzle_bytes)
{
    EncodeTiled fn = encoder();
    if (fn == nullptr) return false;
    const cuuint64_t gd[2] = {words, rows};
    const cuuint64_t gs[1] = {(cuuint64_t)words * 4};
    const cuuint32_t bx[2] = {words, box_rows};
    const cuuint32_t es[2] = {1, 1};
    const CUtensorMapSwizzle sw = swizzle_bytes == 64   ? CU_TENSOR_MAP_SWIZZLE_64B
                                  : swizzle_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                        : CU_TENSOR_MAP_SWIZZLE_NONE;
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(base), gd, gs, bx, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace vq
