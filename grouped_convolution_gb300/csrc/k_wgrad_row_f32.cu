// k_wgrad_row_f32.cu -- weight-gradient row-ring instantiations for float (one
// translation unit per dtype so the unrolled kernels compile in parallel).
#include "k_wgrad_row.cuh"

namespace gconv {
int wrow_slices_f32(const Params &p) { return wrow_slices_dtype<float>(p); }
cudaError_t wrow_launch_f32(const Params &p, const void *x, const void *gy, float *ws,
                         cudaStream_t s) {
    return wrow_launch_dtype<float>(p, x, gy, ws, s);
}
}  // namespace gconv
