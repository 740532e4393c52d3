// tma.cu -- host-side tensor map encoding (see tma.cuh).
#include <mutex>

#include "tma.cuh"

namespace gconv {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}
}  // namespace

bool tma_encode_4d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base,
                   const uint64_t dims[4], const uint64_t strides_bytes[3],
                   const uint32_t box[4]) {
    const uint32_t unit[4] = {1, 1, 1, 1};
    return tma_encode_4d_strided(map, dtype, base, dims, strides_bytes, box, unit);
}

bool tma_encode_4d_strided(CUtensorMap *map, CUtensorMapDataType dtype, const void *base,
                           const uint64_t dims[4], const uint64_t strides_bytes[3],
                           const uint32_t box[4], const uint32_t element_strides[4]) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    cuuint64_t gdim[4] = {dims[0], dims[1], dims[2], dims[3]};
    cuuint64_t gstr[3] = {strides_bytes[0], strides_bytes[1], strides_bytes[2]};
    cuuint32_t bdim[4] = {box[0], box[1], box[2], box[3]};
    cuuint32_t estr[4] = {element_strides[0], element_strides[1], element_strides[2],
                          element_strides[3]};
    CUresult r = fn(map, dtype, 4, const_cast<void *>(base), gdim, gstr, bdim, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace gconv
