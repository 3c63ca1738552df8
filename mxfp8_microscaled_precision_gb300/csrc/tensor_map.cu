// tensor_map.cu -- host-side encoding of TMA tensor maps (cuTensorMapEncodeTiled,
// resolved once through the runtime's driver entry-point query so that the
// library does not link the driver library directly).

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "mxq_internal.h"

namespace mxq {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

}  // namespace

bool encode_tensor_map_3d(CUtensorMap* map, const void* base, bool two_byte_elems, uint64_t inner,
                          uint64_t mid, uint64_t outer, uint64_t mid_stride_bytes,
                          uint64_t outer_stride_bytes, uint32_t box_inner, uint32_t box_mid) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || inner == 0 || mid == 0 || outer == 0) return false;
    const cuuint64_t dims[3] = {inner, mid, outer};
    const cuuint64_t strides[2] = {mid_stride_bytes, outer_stride_bytes};
    const cuuint32_t box[3] = {box_inner, box_mid, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return fn(map, two_byte_elems ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
              const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tensor_map_2d(CUtensorMap* map, const void* base, bool two_byte_elems, uint64_t inner,
                          uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner,
                          uint32_t box_outer, bool swizzle_128b) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || inner == 0 || outer == 0) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1u, 1u};
    return fn(map, two_byte_elems ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
              const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle_128b ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// BF16 matrix [rows, cols] with a row stride of ld elements, as the target of
// tiled stores of 32 x 32 boxes from shared memory laid out with the 64-byte
// swizzle (16-byte chunk j of box row r at chunk position j ^ ((r >> 1) & 3)).
bool encode_tensor_map_bf16_store(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                                  uint64_t ld) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || cols == 0 || rows == 0) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {ld * 2};
    const cuuint32_t box[2] = {32u, 32u};
    const cuuint32_t estr[2] = {1u, 1u};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tensor_map_u8_store(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint64_t ld) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || cols == 0 || rows == 0) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {ld};
    const cuuint32_t box[2] = {32u, 32u};
    const cuuint32_t estr[2] = {1u, 1u};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace mxq
