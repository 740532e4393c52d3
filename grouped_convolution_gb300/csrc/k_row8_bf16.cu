// k_row8_bf16.cu -- dw_row8 instantiations for __nv_bfloat16 (one translation unit per
// dtype so the unrolled kernels compile in parallel).
#include "k_row8.cuh"

namespace gconv {
cudaError_t row8_launch_bf16(const Params &p, const Ptrs &q, cudaStream_t s) {
    return row8_launch_dtype<__nv_bfloat16>(p, q, s);
}
}  // namespace gconv
