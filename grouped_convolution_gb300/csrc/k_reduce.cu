// k_reduce.cu -- grp_reduce: a parallel reduction over the taps for
// convolutions with few outputs (executorch PR #25085, description, second
// paragraph, names this schedule: the taps of one output are summed in
// parallel, for calls with few outputs).
//
// Each output element is shared by L lanes of a warp (L = 8, or 32 when the
// tap count Cin_g*KH*KW is large): lane l accumulates taps l, l+L, l+2L, ...
// in fp32, reading x and w through their strides (any layout), and the L
// partial sums are combined with xor shuffles.  Outputs are numbered in y's
// memory order, so each group of lanes stores next to the previous group.
// It takes every call (any dilation, forward or transposed: the transposed
// gather of executorch PR #25091, description, second paragraph) and pays
// off when there are too few outputs to give each thread its own (a small
// image or channel count with a big kernel).
#include "device_common.cuh"
#include "gconv_internal.h"
#include "launch.cuh"

namespace gconv {
namespace {

constexpr int kReduceThreads = 256;

template <typename T, int L, bool TR>
__global__ void __launch_bounds__(kReduceThreads)
reduce_kernel(const T *__restrict__ x, const T *__restrict__ w, const T *__restrict__ b,
              T *__restrict__ y, Params p, int64_t total) {
    // Let the next kernel in the stream start launching; wait for the
    // previous kernel's memory before reading global memory.
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x % L;
    const int64_t per_block = kReduceThreads / L;
    const int taps = p.Cin_g * p.KH * p.KW;
    const int khw = p.KH * p.KW;
    // The loop runs per warp (base is the same for all its lanes), so every
    // lane reaches the shuffles; groups past the end only skip their store.
    const int64_t warp_base = (int64_t)blockIdx.x * per_block + (threadIdx.x / 32) * (32 / L);
    const int group = (threadIdx.x % 32) / L;
    for (int64_t base = warp_base; base < total; base += (int64_t)gridDim.x * per_block) {
        const int64_t idx = base + group;
        const bool valid = idx < total;
        int64_t r = valid ? idx : 0;
        int n, co, oh, ow;
        if (p.layout == GCONV_LAYOUT_NCHW) {
            ow = (int)(r % p.OW); r /= p.OW;
            oh = (int)(r % p.OH); r /= p.OH;
            co = (int)(r % p.C_out); n = (int)(r / p.C_out);
        } else {
            co = (int)(r % p.C_out); r /= p.C_out;
            ow = (int)(r % p.OW); r /= p.OW;
            oh = (int)(r % p.OH); n = (int)(r / p.OH);
        }
        const int g = co / p.Cout_g;
        const T *xn = x + (int64_t)n * p.xs[0] + (int64_t)g * p.Cin_g * p.xs[1];
        // Weight of (co, ci): w[co, ci] forward, w[g*Cin_g + ci, co - g*Cout_g]
        // transposed.
        const T *wc = TR ? w + (int64_t)g * p.Cin_g * p.ws[0] + (int64_t)(co - g * p.Cout_g) * p.ws[1]
                         : w + (int64_t)co * p.ws[0];
        const int64_t wci = TR ? p.ws[0] : p.ws[1];
        float acc = 0.f;
        for (int tap = lane; valid && tap < taps; tap += L) {
            const int ci = tap / khw, k = tap - ci * khw;
            const int kh = k / p.KW, kw = k - kh * p.KW;
            const int ih = tap_input<TR>(oh, kh, p.sh, p.pbh, p.dh, p.H);
            const int iw = tap_input<TR>(ow, kw, p.sw, p.pbw, p.dw, p.W);
            if (ih >= 0 && iw >= 0) {
                const float xv = load_f32(xn + ci * p.xs[1] + ih * p.xs[2] + iw * p.xs[3]);
                const float wv = load_f32(wc + ci * wci + kh * p.ws[2] + kw * p.ws[3]);
                acc = fmaf(wv, xv, acc);
            }
        }
#pragma unroll
        for (int off = L / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, L);
        if (valid && lane == 0) {
            if (p.has_bias) acc += load_f32(b + (int64_t)co * p.bs);
            y[idx] = from_f32<T>(acc);
        }
    }
}

bool reduce_supports(const gconv_desc &, const Ptrs &) { return true; }

cudaError_t reduce_launch(const Params &p, const Ptrs &q, cudaStream_t s, int *launches) {
    const int64_t total = (int64_t)p.N * p.C_out * p.OH * p.OW;
    const int taps = p.Cin_g * p.KH * p.KW;
    const bool wide = taps >= 128;
    const int L = wide ? 32 : 8;
    int64_t blocks = (total * L + kReduceThreads - 1) / kReduceThreads;
    if (blocks > 152 * 32) blocks = 152 * 32;
    *launches = 1;
    return GCONV_DISPATCH_DTYPE(p.dtype, T, [&] {
        const T *x = static_cast<const T *>(q.x);
        const T *w = static_cast<const T *>(q.w);
        const T *b = static_cast<const T *>(q.b);
        T *y = static_cast<T *>(q.y);
        cudaError_t e;
        auto go = [&](auto kernel) {
            return launch_kernel(kernel, dim3((unsigned)blocks), dim3(kReduceThreads), 0, s, x, w, b,
                              y, p, total);
        };
        if (p.transposed)
            e = wide ? go(reduce_kernel<T, 32, true>) : go(reduce_kernel<T, 8, true>);
        else
            e = wide ? go(reduce_kernel<T, 32, false>) : go(reduce_kernel<T, 8, false>);
        return e != cudaSuccess ? e : cudaGetLastError();
    });
}

}  // namespace

const Schedule kGrpReduce = {"grp_reduce", reduce_supports, reduce_launch};

}  // namespace gconv
