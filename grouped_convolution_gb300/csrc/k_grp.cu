// k_grp.cu -- the grp_plane schedule: which calls it takes and its launcher.
// The kernel is in k_grp.cuh; its instantiations are in k_grp_<dtype>.cu.
#include "k_grp.cuh"

namespace gconv {
namespace {

bool grp_supports(const gconv_desc &d, const Ptrs &q) {
    if (!plain_forward(d)) return false;                    // dilation 1, forward
    (void)q;
    if (d.stride[1] != 1 && d.stride[1] != 2) return false;
    Params p = make_params(d);
    GrpGeom g;
    int cip, mb;
    if (!grp_geometry(p, dtype_size(d.dtype), g, cip, mb)) return false;
    return g.tiles <= INT32_MAX;
}

cudaError_t grp_launch(const Params &p, const Ptrs &q, cudaStream_t s, int *launches) {
    *launches = 1;
    switch (p.dtype) {
    case GCONV_F32: return grp_launch_f32(p, q, s);
    case GCONV_F16: return grp_launch_f16(p, q, s);
    case GCONV_BF16: return grp_launch_bf16(p, q, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

const Schedule kGrpPlane = {"grp_plane", grp_supports, grp_launch};

}  // namespace gconv
