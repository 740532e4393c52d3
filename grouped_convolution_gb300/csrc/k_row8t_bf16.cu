// k_row8t_bf16.cu -- dw_row8 transposed-form instantiations for __nv_bfloat16 (one
// translation unit per dtype so the unrolled kernels compile in parallel).
#include "k_row8t.cuh"

namespace gconv {
cudaError_t row8t_launch_bf16(const Params &p, const Ptrs &q, cudaStream_t s) {
    return row8t_launch_dtype<__nv_bfloat16>(p, q, s);
}
}  // namespace gconv
