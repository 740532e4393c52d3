// k_row8_f32.cu -- dw_row8 instantiations for float (one translation unit per
// dtype so the unrolled kernels compile in parallel).
#include "k_row8.cuh"

namespace gconv {
cudaError_t row8_launch_f32(const Params &p, const Ptrs &q, cudaStream_t s) {
    return row8_launch_dtype<float>(p, q, s);
}
}  // namespace gconv
