// Tensor maps over the pre-tiled fp16 operand arrays, for TMA copies of one
// 128 x 64 chunk at a time.  The array is viewed as a 2-D tensor of `rows`
// rows of 64 fp16 (128 bytes per row, contiguous); a box of 64 x 128 is one
// 16 KB chunk.  The bytes are already in the tensor core's swizzled order, so
// the map itself does no swizzling, and the x coordinate of every copy is 0.
#include "fs_host.cuh"
#include "fs_tc_kernels.cuh"

#include <cuda.h>

#include <mutex>

namespace fs {

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::mutex g_tmap_mu;
EncodeTiledFn g_encode = nullptr;

fs_status encode_fn(EncodeTiledFn* out) {
    std::lock_guard<std::mutex> lk(g_tmap_mu);
    if (g_encode == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) {
            cudaGetLastError();
            return fail(FS_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
        }
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    *out = g_encode;
    return FS_OK;
}

}  // namespace

fs_status make_chunk_tmap(void* map128, const void* base, uint64_t rows) {
    EncodeTiledFn enc = nullptr;
    FS_TRY(encode_fn(&enc));
    const cuuint64_t dims[2] = {64, rows};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {64, 128};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(reinterpret_cast<CUtensorMap*>(map128), CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                     const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FS_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return FS_OK;
}

}  // namespace fs
