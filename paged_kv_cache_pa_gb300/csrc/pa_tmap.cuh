// pa_tmap.cuh -- host-side encoding of TMA tensor maps (cuTensorMapEncodeTiled,
// reached through the runtime's driver entry point, so the library does not
// link the driver library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "pa.h"

namespace pa {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn tmap_encoder() {
    static std::atomic<void *> fn{nullptr};
    void *f = fn.load(std::memory_order_acquire);
    if (!f) {
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !f)
            return nullptr;
        fn.store(f, std::memory_order_release);
    }
    return reinterpret_cast<EncodeTiledFn>(f);
}

// A tiled map of an fp32, fp16 or bf16 tensor with `rank` dimensions
// (innermost first), byte strides of dimensions 1.. , a box, and the 128-byte
// swizzle; reads outside the tensor return zeros, stores outside it are
// dropped.
inline bool encode_tiled(CUtensorMap *map, const void *base, pa_dtype_t dtype, int rank,
                         const cuuint64_t *dims, const cuuint64_t *strides,
                         const cuuint32_t *box) {
    EncodeTiledFn enc = tmap_encoder();
    if (!enc) return false;
    const cuuint32_t elem_strides[5] = {1u, 1u, 1u, 1u, 1u};
    const CUtensorMapDataType ty = dtype == PA_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : dtype == PA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    return enc(map, ty, (cuuint32_t)rank, const_cast<void *>(base), dims, strides, box,
               elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace pa
