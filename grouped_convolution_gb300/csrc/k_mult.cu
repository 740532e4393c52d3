// k_mult.cu -- the dw_mult schedule: which calls it takes and its launcher.
// The kernel is in k_mult.cuh.
#include "k_mult.cuh"

namespace gconv {
namespace {

bool mult_supports(const gconv_desc &d, const Ptrs &q) {
    if (!plain_forward(d)) return false;                    // dilation 1, forward
    if (d.Cin_g != 1 || d.Cout_g > 16) return false;
    if (d.layout != GCONV_LAYOUT_NCHW) return false;
    if (d.KW > kMultMaxKW) return false;
    if (d.stride[1] != 1 && d.stride[1] != 2) return false;
    // x must have unit stride along W (NCHW order guarantees it); x that a
    // tensor map cannot describe is staged with plain loads.
    if (d.x_strides[3] != 1) return false;
    const int es = dtype_size(d.dtype);
    (void)q;
    Params p = make_params(d);
    MultGeom g;
    if (!mult_geometry(p, es, g)) return false;
    return true;
}

cudaError_t mult_launch(const Params &p, const Ptrs &q, cudaStream_t s, int *launches) {
    *launches = 1;
    switch (p.dtype) {
    case GCONV_F32: return mult_launch_f32(p, q, s);
    case GCONV_F16: return mult_launch_f16(p, q, s);
    case GCONV_BF16: return mult_launch_bf16(p, q, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

const Schedule kDwMult = {"dw_mult", mult_supports, mult_launch};

}  // namespace gconv
