// k_wgrad_row.cu -- the partial pass of the weight / bias gradient for
// channels-last depthwise calls with square 3x3, 5x5 or 7x7 kernels
// (multiplier 1, square stride 1 or 2, dilation 1), on the dw_row8 row ring.
//
// The gradient of tap (kh, kw) of channel c is the sum over every output
// pixel of gy[n, c, oh, ow] * x[n, c, oh*S_H - pad_h + kh, ow*S_W - pad_w + kw]
// (the chain rule applied to the direct-stencil sum; the bias gradient is the
// sum of gy).  It is the forward stencil with the roles of weights and
// outputs exchanged, so it runs on the forward schedule's machinery:
//  - the same flat list of output rows (image, column chunk, output row) per
//    channel chunk, split evenly over persistent CTAs (grid y = channel
//    chunk); a run of consecutive output rows reads its input rows once;
//  - each ring stage carries U input rows (TMA box of the row segment with
//    its halo; the zero fill supplies the padding) and the R = ceil(KH/S_H)
//    gy rows whose first tap row lies in those input rows (second TMA box of
//    the same stage, same mbarrier);
//  - thread (cv, pg) owns VEC channels and S output columns.  When an output
//    row's first tap row arrives, its gy vectors move from shared memory into
//    one of R register sets (zero for rows outside the run); every staged
//    input row is widened once into a window and multiplied into the K*K tap
//    accumulators (fp32 channel pairs, packed fma.rn.f32x2) for each open
//    output row -- the forward's accumulator sets become gy sets, its weights
//    become accumulators;
//  - at the end the CTA adds its pixel groups in shared memory (fixed order)
//    and writes one fp32 partial per (channel, tap) and the bias: CTA x of
//    chunk y is workspace slice x.  The finish kernel of the weight-gradient
//    pass adds the slices in a fixed order, so results are reproducible.
//  - Waits are bounded as in the forward: a wait that gives up poisons the
//    thread's accumulators with NaN and stops the ring; the CTA then writes
//    NaN partials without reusing the ring's shared memory.
#include "k_wgrad_row.cuh"

namespace gconv {

int wgrad_row_slices(const Params &p) {
    if (p.transposed || p.Cin_g != 1 || p.Cout_g != 1) return 0;
    if (p.KH != p.KW || p.dh != 1 || p.dw != 1) return 0;
    if (p.KH != 3 && p.KH != 5 && p.KH != 7) return 0;
    if ((p.sh != 1 && p.sh != 2) || p.sw != p.sh) return 0;
    if (p.xs[1] != 1 || p.ys[1] != 1) return 0;   // channels contiguous
    const int64_t es = dtype_size(p.dtype);
    const int vec = p.dtype == GCONV_F32 ? row8_vec<float>(p.KH) : row8_vec<__half>(p.KH);
    if (p.C_out % vec) return 0;
    // TMA: strides in 16-byte units.
    for (int i : {0, 2, 3})
        if ((p.xs[i] * es) % 16 || (p.ys[i] * es) % 16) return 0;
    if (p.N <= 0 || p.OH <= 0 || p.OW <= 0) return 0;
    switch (p.dtype) {
    case GCONV_F32: return wrow_slices_f32(p);
    case GCONV_F16: return wrow_slices_f16(p);
    case GCONV_BF16: return wrow_slices_bf16(p);
    }
    return 0;
}

bool wgrad_row_pointers(const void *x, const void *gy) { return aligned(x, 16) && aligned(gy, 16); }

cudaError_t wgrad_row_partial(const Params &p, const void *x, const void *gy, float *ws,
                              cudaStream_t s) {
    switch (p.dtype) {
    case GCONV_F32: return wrow_launch_f32(p, x, gy, ws, s);
    case GCONV_F16: return wrow_launch_f16(p, x, gy, ws, s);
    case GCONV_BF16: return wrow_launch_bf16(p, x, gy, ws, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gconv
