// Host helper: encode TMA tensor maps through the driver entry point (no
// link-time dependency on libcuda).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.h"

namespace mla {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_once;

void* entry_point(const char* name, int version) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &fn, version, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return fn;
    return nullptr;
}
}  // namespace

unsigned long long current_context_id() {
    std::call_once(g_ctx_once, [] {
        g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(
            entry_point("cuCtxGetCurrent", 4000));
        g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(entry_point("cuCtxGetId", 12000));
    });
    if (!g_ctx_current || !g_ctx_id) return 0;
    CUcontext c = nullptr;
    if (g_ctx_current(&c) != CUDA_SUCCESS || c == nullptr) return 0;
    unsigned long long id = 0;
    return g_ctx_id(c, &id) == CUDA_SUCCESS ? id : 0;
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}
}  // namespace

cudaError_t encode_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                                uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
    if (!encoder()) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_tmap_3d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t mid,
                                uint64_t outer, uint64_t mid_bytes, uint64_t outer_bytes,
                                uint32_t box_inner, uint32_t box_mid, uint32_t box_outer) {
    if (!encoder()) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {inner, mid, outer};
    const cuuint64_t strides[2] = {mid_bytes, outer_bytes};
    const cuuint32_t box[3] = {box_inner, box_mid, box_outer};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                              uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
    if (!encoder()) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace mla
