// k_wgrad_row_bf16.cu -- weight-gradient row-ring instantiations for __nv_bfloat16 (one
// translation unit per dtype so the unrolled kernels compile in parallel).
#include "k_wgrad_row.cuh"

namespace gconv {
int wrow_slices_bf16(const Params &p) { return wrow_slices_dtype<__nv_bfloat16>(p); }
cudaError_t wrow_launch_bf16(const Params &p, const void *x, const void *gy, float *ws,
                         cudaStream_t s) {
    return wrow_launch_dtype<__nv_bfloat16>(p, x, gy, ws, s);
}
}  // namespace gconv
