// tmap.cuh -- host-side creation of TMA tensor maps (cuTensorMapEncodeTiled,
// fetched through the runtime's driver entry-point query so the library does not
// link libcuda directly).
#pragma once

#include "common.cuh"

namespace moe {

// Encode a tiled tensor map of `rank` dimensions (innermost first).  strides_bytes
// holds rank-1 byte strides of dimensions 1..rank-1.  Returns false on failure.
inline bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base,
                        const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                        CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    using EncodeFn = decltype(&cuTensorMapEncodeTiled);
    static EncodeFn fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !p)
            return false;
        fn = reinterpret_cast<EncodeFn>(p);
    }
    uint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(map, dt, (cuuint32_t)rank, const_cast<void*>(base), (const cuuint64_t*)dims,
                    (const cuuint64_t*)strides_bytes, (const cuuint32_t*)box, (const cuuint32_t*)estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace moe
