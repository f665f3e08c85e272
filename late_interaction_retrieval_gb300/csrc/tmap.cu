// tmap.cu -- host-side TMA tensor-map encoding for the tensor-core kernels.
//
// cuTensorMapEncodeTiled is a driver entry point; it is resolved once through
// the runtime (cudaGetDriverEntryPointByVersion) so that the library links
// only against the CUDA runtime and loads on machines without a driver.
#include <mutex>

#include <cuda.h>

#include "tmap.h"

namespace lik {

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::once_flag g_once;
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn encoder() {
    std::call_once(g_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    });
    return g_encode;
}

}  // namespace

bool encode_tmap_kmajor(CUtensorMap* map, int dtype, const void* base, int rank,
                        const uint64_t* dims, const uint64_t* strides_bytes,
                        const uint32_t* box) {
    EncodeTiledFn fn = encoder();
    if (!fn) return false;
    cuuint64_t gdim[3], gstride[2];
    cuuint32_t bdim[3], estride[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        gdim[i] = dims[i];
        bdim[i] = box[i];
    }
    for (int i = 0; i + 1 < rank; ++i) gstride[i] = strides_bytes[i];
    const CUtensorMapDataType t = dtype == kBF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                  : dtype == kF32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult r = fn(map, t, static_cast<cuuint32_t>(rank), const_cast<void*>(base), gdim, gstride,
                    bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace lik
