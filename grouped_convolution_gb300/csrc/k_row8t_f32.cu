// k_row8t_f32.cu -- dw_row8 transposed-form instantiations for float (one
// translation unit per dtype so the unrolled kernels compile in parallel).
#include "k_row8t.cuh"

namespace gconv {
cudaError_t row8t_launch_f32(const Params &p, const Ptrs &q, cudaStream_t s) {
    return row8t_launch_dtype<float>(p, q, s);
}
}  // namespace gconv
