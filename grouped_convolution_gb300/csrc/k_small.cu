// k_small.cu -- dw_small: depthwise convolution (one input channel per
// group, any multiplier) of problems too small for a persistent staged
// kernel to pay off, in one pass with no shared memory and no barrier.
//
// The operation is the depthwise case of the direct stencil of executorch
// PR #25085 (description, second paragraph); the schedule is this library's
// own.  On a problem of a few hundred thousand outputs a persistent kernel
// with a TMA ring spends its time filling and draining the ring; here every
// thread issues all of its loads at once and the whole problem is a single
// wave of threads:
//  - A thread computes 4 consecutive outputs of one output row of one
//    output channel; threads are numbered in (image, channel, row, column
//    quad) order, so a warp's loads and stores fall on few cache lines in
//    NCHW-ordered tensors (any other strides are still correct).
//  - Square 3x3, 5x5 and 7x7 kernels at stride 1 and dilation 1 along the
//    row: every input value and weight the thread needs is loaded at once
//    (K rows of 3 + K values, K*K weights), so the thread waits for memory
//    once; other shapes loop over the taps, loading each tap of each output
//    on its own (the L1 cache catches the overlap).
//  - fp32 accumulation in (kh, kw) order, the bias added in fp32, one
//    rounding to the output dtype.

#include "device_common.cuh"
#include "gconv_internal.h"
#include "launch.cuh"

#include <utility>

namespace gconv {
namespace {

// Launched without programmatic dependent launch: measured on the 3x3
// layer of 1x32x56x56, a launch that waits for the previous kernel at
// griddepcontrol.wait took 4.1 us against 3.0 us for a plain launch (the
// persistent kernels, whose prologue overlaps the previous kernel, gain
// from it instead).
template <typename... KArgs, typename... Args>
cudaError_t launch_plain(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t s,
                         Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

constexpr int kSmallQuad = 4;     // outputs per thread
constexpr int kSmallThreads = 256;

// Four consecutive outputs rounded and stored at once: y + ow0 is aligned
// to the quad's size (checked on the host).
__device__ __forceinline__ void store_quad(float *q, float a, float b, float c, float d) {
    *reinterpret_cast<float4 *>(q) = make_float4(a, b, c, d);
}
template <typename T>
__device__ __forceinline__ void store_quad(T *q, float a, float b, float c, float d) {
    uint2 o;
    o.x = pack2(a, b, (T *)nullptr);
    o.y = pack2(c, d, (T *)nullptr);
    *reinterpret_cast<uint2 *>(q) = o;
}

// Square K x K kernel, stride 1 and dilation 1 along the row (any stride
// and dilation down the column).
template <typename T, int K>
__global__ void __launch_bounds__(kSmallThreads)
small_kernel_k(const T *__restrict__ x, const T *__restrict__ w, const T *__restrict__ b,
               T *__restrict__ y, Params p, int quads, int64_t total, int vec) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t idx = (int64_t)blockIdx.x * kSmallThreads + threadIdx.x;
    if (idx >= total) return;
    int r = (int)(idx / quads);
    const int q = (int)(idx - (int64_t)r * quads);
    const int oh = r % p.OH;
    r /= p.OH;
    const int co = r % p.C_out;
    const int n = r / p.C_out;
    const int ci = co / p.Cout_g;   // one input channel per group
    const T *xc = x + (int64_t)n * p.xs[0] + (int64_t)ci * p.xs[1];
    const T *wc = w + (int64_t)co * p.ws[0];
    const int ow0 = q * kSmallQuad;
    const int iw0 = ow0 - p.pbw;
    constexpr int WIN = kSmallQuad - 1 + K;
    float win[K][WIN];
    float wr[K][K];
#pragma unroll
    for (int kh = 0; kh < K; ++kh) {
        const int ih = oh * p.sh - p.pbh + kh * p.dh;
        const bool row_ok = ih >= 0 && ih < p.H;
        const T *row = xc + (int64_t)(row_ok ? ih : 0) * p.xs[2];
#pragma unroll
        for (int j = 0; j < WIN; ++j) {
            const int iw = iw0 + j;
            win[kh][j] = (row_ok && iw >= 0 && iw < p.W) ? load_f32(row + (int64_t)iw * p.xs[3]) : 0.f;
        }
#pragma unroll
        for (int kw = 0; kw < K; ++kw)
            wr[kh][kw] = load_f32(wc + (int64_t)kh * p.ws[2] + (int64_t)kw * p.ws[3]);
    }
    float acc[kSmallQuad] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kh = 0; kh < K; ++kh)
#pragma unroll
        for (int kw = 0; kw < K; ++kw)
#pragma unroll
            for (int i = 0; i < kSmallQuad; ++i) acc[i] = fmaf(wr[kh][kw], win[kh][i + kw], acc[i]);
    const float bv = p.has_bias ? load_f32(b + (int64_t)co * p.bs) : 0.f;
    T *yr = y + (int64_t)n * p.ys[0] + (int64_t)co * p.ys[1] + (int64_t)oh * p.ys[2];
    if (vec && ow0 + kSmallQuad <= p.OW) {
        // the quad's 4 outputs in one store (16 bytes fp32, 8 bytes 16-bit)
        store_quad(yr + ow0, acc[0] + bv, acc[1] + bv, acc[2] + bv, acc[3] + bv);
    } else {
#pragma unroll
        for (int i = 0; i < kSmallQuad; ++i)
            if (ow0 + i < p.OW) yr[(int64_t)(ow0 + i) * p.ys[3]] = from_f32<T>(acc[i] + bv);
    }
}

// Any other shape: a loop over the taps.
template <typename T, bool UNIT>
__global__ void __launch_bounds__(kSmallThreads)
small_kernel(const T *__restrict__ x, const T *__restrict__ w, const T *__restrict__ b,
             T *__restrict__ y, Params p, int quads, int64_t total) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t idx = (int64_t)blockIdx.x * kSmallThreads + threadIdx.x;
    if (idx >= total) return;
    int r = (int)(idx / quads);
    const int q = (int)(idx - (int64_t)r * quads);
    const int oh = r % p.OH;
    r /= p.OH;
    const int co = r % p.C_out;
    const int n = r / p.C_out;
    const int ci = co / p.Cout_g;   // one input channel per group
    const T *xc = x + (int64_t)n * p.xs[0] + (int64_t)ci * p.xs[1];
    const T *wc = w + (int64_t)co * p.ws[0];
    const int ow0 = q * kSmallQuad;
    float acc[kSmallQuad] = {0.f, 0.f, 0.f, 0.f};
    for (int kh = 0; kh < p.KH; ++kh) {
        const int ih = oh * p.sh - p.pbh + kh * p.dh;
        if (ih < 0 || ih >= p.H) continue;
        const T *row = xc + (int64_t)ih * p.xs[2];
        if (UNIT) {
            // input columns ow0 - pbw .. ow0 - pbw + 3 + KW - 1
            const int iw0 = ow0 - p.pbw;
            float win[kSmallQuad - 1 + 9];
#pragma unroll
            for (int j = 0; j < kSmallQuad - 1 + 9; ++j) {
                const int iw = iw0 + j;
                win[j] = (j < kSmallQuad - 1 + p.KW && iw >= 0 && iw < p.W)
                             ? load_f32(row + (int64_t)iw * p.xs[3])
                             : 0.f;
            }
#pragma unroll
            for (int kw = 0; kw < 9; ++kw) {
                if (kw >= p.KW) break;
                const float wv = load_f32(wc + (int64_t)kh * p.ws[2] + (int64_t)kw * p.ws[3]);
#pragma unroll
                for (int i = 0; i < kSmallQuad; ++i) acc[i] = fmaf(wv, win[i + kw], acc[i]);
            }
        } else {
            for (int kw = 0; kw < p.KW; ++kw) {
                const float wv = load_f32(wc + (int64_t)kh * p.ws[2] + (int64_t)kw * p.ws[3]);
#pragma unroll
                for (int i = 0; i < kSmallQuad; ++i) {
                    const int iw = (ow0 + i) * p.sw - p.pbw + kw * p.dw;
                    const float xv = (iw >= 0 && iw < p.W) ? load_f32(row + (int64_t)iw * p.xs[3]) : 0.f;
                    acc[i] = fmaf(wv, xv, acc[i]);
                }
            }
        }
    }
    const float bv = p.has_bias ? load_f32(b + (int64_t)co * p.bs) : 0.f;
    T *yr = y + (int64_t)n * p.ys[0] + (int64_t)co * p.ys[1] + (int64_t)oh * p.ys[2];
#pragma unroll
    for (int i = 0; i < kSmallQuad; ++i)
        if (ow0 + i < p.OW) yr[(int64_t)(ow0 + i) * p.ys[3]] = from_f32<T>(acc[i] + bv);
}

bool small_supports(const gconv_desc &d, const Ptrs &) {
    if (d.transposed || d.Cin_g != 1) return false;
    // 32-bit row and channel indices; the thread index is 64-bit
    return (int64_t)d.N * d.C_out * d.OH <= INT32_MAX && d.H <= INT32_MAX / 16 &&
           d.W <= INT32_MAX / 16;
}

cudaError_t small_launch(const Params &p, const Ptrs &q, cudaStream_t s, int *launches) {
    *launches = 1;
    const int quads = (p.OW + kSmallQuad - 1) / kSmallQuad;
    const int64_t total = (int64_t)p.N * p.C_out * p.OH * quads;
    const int64_t blocks = (total + kSmallThreads - 1) / kSmallThreads;
    if (blocks > INT32_MAX) return cudaErrorInvalidValue;
    const bool unit = p.sw == 1 && p.dw == 1;
    const int K = unit && p.KH == p.KW ? p.KH : 0;
    // one vector store per quad: unit column stride, quads aligned in memory
    const int qb = kSmallQuad * (int)dtype_size(p.dtype);
    const int vec = p.ys[3] == 1 && (p.ys[2] * dtype_size(p.dtype)) % qb == 0 &&
                    (p.ys[1] * dtype_size(p.dtype)) % qb == 0 &&
                    (p.ys[0] * dtype_size(p.dtype)) % qb == 0 && aligned(q.y, qb);
    return GCONV_DISPATCH_DTYPE(p.dtype, T, [&] {
        const T *x = static_cast<const T *>(q.x);
        const T *w = static_cast<const T *>(q.w);
        const T *b = static_cast<const T *>(q.b);
        T *y = static_cast<T *>(q.y);
        const dim3 grid((unsigned)blocks), block(kSmallThreads);
        cudaError_t e;
        if (K == 3)
            e = launch_plain(small_kernel_k<T, 3>, grid, block, s, x, w, b, y, p, quads, total, vec);
        else if (K == 5)
            e = launch_plain(small_kernel_k<T, 5>, grid, block, s, x, w, b, y, p, quads, total, vec);
        else if (K == 7)
            e = launch_plain(small_kernel_k<T, 7>, grid, block, s, x, w, b, y, p, quads, total, vec);
        else
            e = unit ? launch_plain(small_kernel<T, true>, grid, block, s, x, w, b, y, p, quads, total)
                     : launch_plain(small_kernel<T, false>, grid, block, s, x, w, b, y, p, quads, total);
        return e != cudaSuccess ? e : cudaGetLastError();
    });
}

}  // namespace

const Schedule kDwSmall = {"dw_small", small_supports, small_launch};

}  // namespace gconv
