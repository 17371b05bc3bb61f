// Host-side helpers of the tensor-core path: TMA descriptor encoding through
// the driver entry point (no link-time dependency on libcuda).
#include <cudaTypedefs.h>

#include <mutex>

#include "tc_common.cuh"

namespace saf {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void load_encode() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    else
        cudaGetLastError();
}

}  // namespace

namespace {
bool make_tmap_3d(CUtensorMap* map, CUtensorMapDataType type, uint64_t elem, const void* base, uint64_t n0,
                  uint64_t n1, uint64_t n2, uint32_t b0, uint32_t b1) {
    std::call_once(g_encode_once, load_encode);
    if (!g_encode) return false;
    const cuuint64_t dims[3] = {n0, n1, n2};
    const cuuint64_t strides[2] = {n0 * elem, n0 * n1 * elem};  // bytes, dims 1 and 2
    const cuuint32_t box[3] = {b0, b1, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = g_encode(map, type, 3, const_cast<void*>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}
}  // namespace

bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, uint64_t n0, uint64_t n1, uint64_t n2, uint32_t b0,
                       uint32_t b1) {
    return make_tmap_3d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, n0, n1, n2, b0, b1);
}

bool make_tmap_f32_3d(CUtensorMap* map, const void* base, uint64_t n0, uint64_t n1, uint64_t n2, uint32_t b0,
                      uint32_t b1) {
    return make_tmap_3d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, n0, n1, n2, b0, b1);
}

}  // namespace saf
