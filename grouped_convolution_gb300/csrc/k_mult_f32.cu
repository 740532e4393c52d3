// k_mult_f32.cu -- dw_mult instantiations for float (one translation unit per
// dtype so the unrolled kernels compile in parallel).
#include "k_mult.cuh"

namespace gconv {
cudaError_t mult_launch_f32(const Params &p, const Ptrs &q, cudaStream_t s) {
    return mult_launch_dtype<float>(p, q, s);
}
}  // namespace gconv
