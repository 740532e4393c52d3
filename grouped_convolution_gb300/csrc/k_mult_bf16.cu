// k_mult_bf16.cu -- dw_mult instantiations for __nv_bfloat16 (one translation unit per
// dtype so the unrolled kernels compile in parallel).
#include "k_mult.cuh"

namespace gconv {
cudaError_t mult_launch_bf16(const Params &p, const Ptrs &q, cudaStream_t s) {
    return mult_launch_dtype<__nv_bfloat16>(p, q, s);
}
}  // namespace gconv
