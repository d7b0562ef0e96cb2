// Host side of the tile loads: tensor maps for the tensor-memory-access unit
// (TMA).  The encoder is a driver entry point, looked up once through the
// runtime, so the library links no driver library of its own.
#include <cuda.h>
#include <cuda_runtime.h>

#include "kernels.h"

namespace gdn {
namespace {

typedef CUresult (*EncodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
    static const EncodeTiled fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiled>(nullptr);
        return reinterpret_cast<EncodeTiled>(p);
    }();
    return fn;
}

}  // namespace

cudaError_t make_rows_map(CUtensorMap* m, const float* base, int heads, int64_t T,
                          int64_t token_stride, bool mn_major) {
    const EncodeTiled enc = encoder();
    if (enc == nullptr) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)kTileCols, (cuuint64_t)heads, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)kTileCols * sizeof(float),
                                   (cuuint64_t)token_stride * sizeof(float)};
    const cuuint32_t box[3] = {32, 1, 64};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           mn_major ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B
                                    : CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace gdn
