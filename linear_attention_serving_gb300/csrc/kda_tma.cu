// kda_tma.cu -- tensor maps of the prefill inputs for the tensor-memory-access
// (TMA) tile loads of the bf16 preparation.
//
// Each input is a [T, H, D] tensor (q, k, v in bf16, z in fp32), described as a
// 3-D tensor of dimensions {D, H, T} so that one tile load fetches the rows of
// one head over one 64-token chunk: box {D, 1, C}.  Rows past the end of the
// tensor come back as zeros; rows of a following document inside the box are
// masked by the kernel.  cuTensorMapEncodeTiled is reached through the
// runtime's driver entry point, so the library keeps no link-time dependency
// on the driver library.
#include <cuda.h>

#include <mutex>

#include "kda_internal.cuh"

namespace kda {

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return (EncodeTiledFn)f;
    }();
    return fn;
}

int encode_rows(CUtensorMap *m, const void *p, CUtensorMapDataType type, uint32_t elem, int64_t T, int H) {
    const cuuint64_t dim[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t stride[2] = {(cuuint64_t)D * elem, (cuuint64_t)H * D * elem};  // bytes, dims 1 and 2
    const cuuint32_t box[3] = {(cuuint32_t)D, 1u, (cuuint32_t)C};
    const cuuint32_t estride[3] = {1u, 1u, 1u};
    const EncodeTiledFn fn = encode_tiled();
    if (!fn) return KDA_ERR_CUDA;
    const CUresult r = fn(m, type, 3, const_cast<void *>(p), dim, stride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace

int make_input_maps(const void *q, const void *k, const void *v, const float *z, int64_t T, int H, InputMaps *out) {
    int rc;
    if ((rc = encode_rows(&out->q, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, H))) return rc;
    if ((rc = encode_rows(&out->k, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, H))) return rc;
    if ((rc = encode_rows(&out->v, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, H))) return rc;
    return encode_rows(&out->z, z, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, T, H);
}

}  // namespace kda
