// k_row8.cu -- the dw_row8 schedule: which calls it takes and its launcher.
// The forward kernel is in k_row8.cuh, the stride-2 transposed one in
// k_row8t.cuh.
#include "k_row8.cuh"
#include "k_row8t.cuh"

namespace gconv {
namespace {

// The transposed form (k_row8t.cuh): stride 2, square 3/5/7 kernels.
bool row8t_supports(const gconv_desc &d, const Ptrs &q) {
    if (d.dilation[0] != 1 || d.dilation[1] != 1) return false;
    if (d.Cin_g != 1 || d.Cout_g != 1) return false;          // multiplier 1
    if (d.layout != GCONV_LAYOUT_NHWC) return false;          // channel-contiguous
    if (d.KH != d.KW) return false;
    if (d.KH != 3 && d.KH != 5 && d.KH != 7) return false;
    if (d.stride[0] != 2 || d.stride[1] != 2) return false;
    const int es = dtype_size(d.dtype);
    const int vec = d.dtype == GCONV_F32 ? row8_vec<float>((int)d.KH) : row8_vec<__half>((int)d.KH);
    if (d.C_out % vec != 0) return false;
    if (!aligned(q.x, 16)) return false;
    if ((d.x_strides[0] * es) % 16 || (d.x_strides[2] * es) % 16 || (d.x_strides[3] * es) % 16)
        return false;
    if (!aligned(q.y, (uintptr_t)(vec * es))) return false;
    Params p = make_params(d);
    if (p.xs[1] != 1 || p.ys[1] != 1) return false;
    switch (d.dtype) {
    case GCONV_F32: return row8t_fits_dtype<float>(p);
    case GCONV_F16: return row8t_fits_dtype<__half>(p);
    case GCONV_BF16: return row8t_fits_dtype<__nv_bfloat16>(p);
    }
    return false;
}

bool row8_supports(const gconv_desc &d, const Ptrs &q) {
    if (d.transposed) return row8t_supports(d, q);
    // Dilation 1, or 2 in both dims for 3x3 kernels at stride 1 (at stride 2
    // every other staged row and column would go unused).
    const bool dil1 = d.dilation[0] == 1 && d.dilation[1] == 1;
    const bool dil2 = d.dilation[0] == 2 && d.dilation[1] == 2 && d.KH == 3 && d.KW == 3 &&
                      d.stride[0] == 1 && d.stride[1] == 1;
    if (!dil1 && !dil2) return false;
    if (d.Cin_g != 1 || d.Cout_g != 1) return false;          // multiplier 1
    if (d.layout != GCONV_LAYOUT_NHWC) return false;          // channel-contiguous
    if (d.KH != d.KW) return false;
    if (d.KH != 3 && d.KH != 5 && d.KH != 7) return false;
    if (d.stride[0] != 1 && d.stride[0] != 2) return false;
    if (d.stride[1] != d.stride[0]) return false;             // square strides
    const int es = dtype_size(d.dtype);
    const int vec = d.dtype == GCONV_F32 ? row8_vec<float>((int)d.KH) : row8_vec<__half>((int)d.KH);
    if (d.C_out % vec != 0) return false;
    // TMA: 16-byte aligned base, strides in 16-byte units, the channel
    // dim contiguous (channels-last order guarantees it).
    if (!aligned(q.x, 16)) return false;
    if ((d.x_strides[0] * es) % 16 || (d.x_strides[2] * es) % 16 || (d.x_strides[3] * es) % 16)
        return false;
    // vector stores
    if (!aligned(q.y, (uintptr_t)(vec * es))) return false;
    Params p = make_params(d);
    switch (d.dtype) {
    case GCONV_F32: return row8_fits_dtype<float>(p);
    case GCONV_F16: return row8_fits_dtype<__half>(p);
    case GCONV_BF16: return row8_fits_dtype<__nv_bfloat16>(p);
    }
    return false;
}

cudaError_t row8_launch(const Params &p, const Ptrs &q, cudaStream_t s, int *launches) {
    *launches = 1;
    if (p.transposed) {
        switch (p.dtype) {
        case GCONV_F32: return row8t_launch_f32(p, q, s);
        case GCONV_F16: return row8t_launch_f16(p, q, s);
        case GCONV_BF16: return row8t_launch_bf16(p, q, s);
        }
        return cudaErrorInvalidValue;
    }
    switch (p.dtype) {
    case GCONV_F32: return row8_launch_f32(p, q, s);
    case GCONV_F16: return row8_launch_f16(p, q, s);
    case GCONV_BF16: return row8_launch_bf16(p, q, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

const Schedule kDwRow8 = {"dw_row8", row8_supports, row8_launch};

}  // namespace gconv
