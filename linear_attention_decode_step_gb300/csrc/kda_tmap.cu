// Tensor maps (the descriptors of tiled tensor copies, cp.async.bulk.tensor)
// encoded on the host. cuTensorMapEncodeTiled is looked up once through the
// runtime's driver entry point, so the library does not link the driver
// library itself.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kda_internal.cuh"

namespace kda {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static const EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

}  // namespace

cudaError_t make_tensor_map(CUtensorMap *map, const void *base, bool bf16, int rank,
                            const uint64_t *dims, const uint32_t *box, bool swizzle128, int l2_promotion) {
    const EncodeTiledFn fn = encode_tiled();
    if (!fn) return cudaErrorNotSupported;
    const uint64_t esz = bf16 ? 2 : 4;
    cuuint64_t gdim[5], gstr[4];
    cuuint32_t bdim[5], estr[5];
    uint64_t stride = esz;
    for (int i = 0; i < rank; ++i) {
        gdim[i] = dims[i];
        bdim[i] = box[i];
        estr[i] = 1;
        if (i > 0) gstr[i - 1] = stride;
        stride *= dims[i];
    }
    const CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                          (cuuint32_t)rank, const_cast<void *>(base), gdim, gstr, bdim, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          l2_promotion == 0   ? CU_TENSOR_MAP_L2_PROMOTION_NONE
                          : l2_promotion == 1 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                              : CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace kda
