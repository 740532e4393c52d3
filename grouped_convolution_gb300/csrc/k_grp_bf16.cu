// k_grp_bf16.cu -- grp_plane instantiations for __nv_bfloat16 (one translation unit per
// dtype so the unrolled kernels compile in parallel).
#include "k_grp_impl.cuh"

namespace gconv {
cudaError_t grp_launch_bf16(const Params &p, const Ptrs &q, cudaStream_t s) {
    return grp_launch_dtype<__nv_bfloat16>(p, q, s);
}
}  // namespace gconv
