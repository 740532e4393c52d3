// k_grp_f32.cu -- grp_plane instantiations for float (one translation unit per
// dtype so the unrolled kernels compile in parallel).
#include "k_grp_impl.cuh"

namespace gconv {
cudaError_t grp_launch_f32(const Params &p, const Ptrs &q, cudaStream_t s) {
    return grp_launch_dtype<float>(p, q, s);
}
}  // namespace gconv
