// tmap.h -- host-side encoding of TMA tensor maps through the driver entry point (the library
// does not link libcuda; the runtime hands out the driver function).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gemma {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// bf16 tensor of `rank` dims (innermost first), byte strides of dims 1..rank-1, box sizes and
// a shared-memory swizzle; out-of-bounds elements read as zero (and are not written by stores).
// Returns false on failure.
inline bool encode_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                        const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle swizzle) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    uint32_t elem_strides[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank,
                     const_cast<void*>(base), reinterpret_cast<const cuuint64_t*>(dims),
                     reinterpret_cast<const cuuint64_t*>(strides),
                     reinterpret_cast<const cuuint32_t*>(box), elem_strides,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}
// the same with the 128-byte swizzle (rows of 64 bf16)
inline bool encode_bf16_sw128(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                              const uint64_t* strides, const uint32_t* box) {
    return encode_bf16(map, base, rank, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace gemma
