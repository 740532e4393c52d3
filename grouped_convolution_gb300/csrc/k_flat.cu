// k_flat.cu -- dw_flat, the schedule that takes every call (executorch PR
// #25085, description, second paragraph, names it as the fallback).
//
// One thread per output element, threads numbered in y's memory order so
// stores are coalesced in either layout.  x, w and bias are read through
// their strides, so every layout, group shape (Cin_g <= 8, any Cout_g),
// multiplier and dilation runs here, forward or transposed (the transposed
// gather of executorch PR #25091, description, second paragraph, with the
// [C_in, Cout_g, KH, KW] weight); the specialised schedules cover the hot
// shapes.
// Accumulation is fp32 in (ci, kh, kw) order; the epilogue adds the bias and
// rounds once to the output dtype.

#include "device_common.cuh"
#include "gconv_internal.h"
#include "launch.cuh"

namespace gconv {
namespace {

template <typename T, typename I, bool TR>
__global__ void __launch_bounds__(256)
flat_kernel(const T *__restrict__ x, const T *__restrict__ w, const T *__restrict__ b,
            T *__restrict__ y, Params p, int64_t total) {
    // Let the next kernel in the stream start launching; wait for the
    // previous kernel's memory before reading global memory.
    pdl_launch_dependents();
    pdl_wait();
    const I OW = p.OW, OH = p.OH, Co = p.C_out;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        // Decompose the linear index in y's memory order.
        I n, co, oh, ow;
        I r = (I)idx;
        if (p.layout == GCONV_LAYOUT_NCHW) {
            ow = r % OW; r /= OW;
            oh = r % OH; r /= OH;
            co = r % Co; n = r / Co;
        } else {
            co = r % Co; r /= Co;
            ow = r % OW; r /= OW;
            oh = r % OH; n = r / OH;
        }
        const int g = (int)(co / p.Cout_g);
        const T *xn = x + (int64_t)n * p.xs[0] + (int64_t)g * p.Cin_g * p.xs[1];
        // Weight of (co, ci): w[co, ci] forward, w[g*Cin_g + ci, co - g*Cout_g]
        // transposed.
        const T *wc = TR ? w + (int64_t)g * p.Cin_g * p.ws[0] + (int64_t)(co - g * p.Cout_g) * p.ws[1]
                         : w + (int64_t)co * p.ws[0];
        const int64_t wci = TR ? p.ws[0] : p.ws[1];
        float acc = 0.f;
        for (int ci = 0; ci < p.Cin_g; ++ci) {
            for (int kh = 0; kh < p.KH; ++kh) {
                const int ih = tap_input<TR>((int)oh, kh, p.sh, p.pbh, p.dh, p.H);
                if (ih < 0) continue;
                for (int kw = 0; kw < p.KW; ++kw) {
                    const int iw = tap_input<TR>((int)ow, kw, p.sw, p.pbw, p.dw, p.W);
                    if (iw < 0) continue;
                    const float xv = load_f32(xn + ci * p.xs[1] + ih * p.xs[2] + iw * p.xs[3]);
                    const float wv = load_f32(wc + ci * wci + kh * p.ws[2] + kw * p.ws[3]);
                    acc = fmaf(wv, xv, acc);
                }
            }
        }
        if (p.has_bias) acc += load_f32(b + (int64_t)co * p.bs);
        y[idx] = from_f32<T>(acc);
    }
}

bool flat_supports(const gconv_desc &, const Ptrs &) { return true; }

cudaError_t flat_launch(const Params &p, const Ptrs &q, cudaStream_t s, int *launches) {
    const int64_t total = (int64_t)p.N * p.C_out * p.OH * p.OW;
    const int64_t per_image = (int64_t)p.C_out * p.OH * p.OW;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    if (blocks > 152 * 64) blocks = 152 * 64;   // grid-stride beyond 64 blocks per SM
    return GCONV_DISPATCH_DTYPE(p.dtype, T, [&] {
        const T *x = static_cast<const T *>(q.x);
        const T *w = static_cast<const T *>(q.w);
        const T *b = static_cast<const T *>(q.b);
        T *y = static_cast<T *>(q.y);
        cudaError_t e;
        const bool small = total <= INT32_MAX;
        if (p.transposed)
            e = small ? launch_kernel(flat_kernel<T, int, true>, dim3((unsigned)blocks), dim3(threads),
                                   0, s, x, w, b, y, p, total)
                      : launch_kernel(flat_kernel<T, int64_t, true>, dim3((unsigned)blocks),
                                   dim3(threads), 0, s, x, w, b, y, p, total);
        else
            e = small ? launch_kernel(flat_kernel<T, int, false>, dim3((unsigned)blocks),
                                   dim3(threads), 0, s, x, w, b, y, p, total)
                      : launch_kernel(flat_kernel<T, int64_t, false>, dim3((unsigned)blocks),
                                   dim3(threads), 0, s, x, w, b, y, p, total);
        (void)per_image;
        *launches = 1;
        return e != cudaSuccess ? e : cudaGetLastError();
    });
}

}  // namespace

const Schedule kDwFlat = {"dw_flat", flat_supports, flat_launch};

}  // namespace gconv
