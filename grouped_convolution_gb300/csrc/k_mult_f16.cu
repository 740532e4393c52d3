// k_mult_f16.cu -- dw_mult instantiations for __half (one translation unit per
// dtype so the unrolled kernels compile in parallel).
#include "k_mult.cuh"

namespace gconv {
cudaError_t mult_launch_f16(const Params &p, const Ptrs &q, cudaStream_t s) {
    return mult_launch_dtype<__half>(p, q, s);
}
}  // namespace gconv
