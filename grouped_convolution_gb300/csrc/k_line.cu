// k_line.cu -- dw_line: channels-last depthwise convolution (one input and
// one output channel per group) for the shapes dw_row8 does not take: 1-D
// sequences (the height-1 case), non-square or 9x9 kernels, strides above 2,
// any dilation, and the transposed gather of executorch PR #25091
// "Run transposed convolutions on the implicit-GEMM template" (description,
// second paragraph: output o reads input (o + pad_before - k*d) / stride
// when that is a whole number inside the input).
//
// Design: a block owns one chunk of CVb consecutive 16-byte channel vectors
// (blockIdx.y) and walks strips of S consecutive output pixels of one output
// row (grid-stride over blockIdx.x).  Lane (cv, strip): cv fastest, so the
// lanes of a warp read and write consecutive 16-byte vectors of one pixel
// (fully used 32-byte sectors).  The chunk's KH*KW weights and its bias sit
// in shared memory as fp32 [tap][channel] and are read as broadcast vectors;
// input vectors are read straight from global memory (the other taps' reads
// of a pixel hit L1), widened once per read, and multiplied into fp32
// accumulators with packed FMAs; one rounding per output at the store.
#include "device_common.cuh"
#include "gconv_internal.h"
#include "launch.cuh"
#include "stencil_math.cuh"

namespace gconv {
namespace {

constexpr int kLineThreads = 256;
constexpr int kLineS = 4;   // output pixels per lane

template <typename T> constexpr int line_vec() { return 16 / (int)sizeof(T); }

struct LineGeom {
    int CV;      // channel vectors in the tensor
    int CVb;     // channel vectors per block (lanes along channels)
    int PB;      // strips per block pass (lanes along pixels)
    int NSW;     // strips per output row
    int64_t items;   // N * OH * NSW
};

bool line_geometry(const Params &p, int es, LineGeom &g) {
    const int vec = 16 / es;
    if (p.C_out % vec != 0) return false;
    g.CV = p.C_out / vec;
    g.CVb = g.CV < 32 ? g.CV : 32;
    g.PB = kLineThreads / g.CVb;
    g.NSW = (p.OW + kLineS - 1) / kLineS;
    g.items = (int64_t)p.N * p.OH * g.NSW;
    return g.CV >= 1;
}

template <typename T, bool TR>
__global__ void __launch_bounds__(kLineThreads)
line_kernel(const T *__restrict__ x, const T *__restrict__ w, const T *__restrict__ b,
            T *__restrict__ y, Params p, LineGeom g) {
    // Let the next kernel in the stream start launching; wait for the
    // previous kernel's memory before reading global memory.
    pdl_launch_dependents();
    pdl_wait();
    constexpr int VEC = line_vec<T>();
    constexpr int P = VEC / 2;
    constexpr int S = kLineS;
    using V = Vec<T, VEC>;
    using IO = VecIO<16>;
    extern __shared__ __align__(16) float line_w[];   // [KH*KW + 1][CVb * VEC]

    const int taps = p.KH * p.KW;
    const int cb = g.CVb * VEC;                  // channels per block
    const int c_first = blockIdx.y * cb;
    const int t = threadIdx.x;
    // Stage the chunk's weights (w[c, 0, kh, kw], or w[c, 0, ...] of the
    // transposed [C_in, 1, KH, KW] weight: the same element) and bias.
    for (int e = t; e < (taps + 1) * cb; e += blockDim.x) {
        const int tap = e / cb, cl = e - tap * cb, c = c_first + cl;
        float v = 0.f;
        if (c < p.C_out) {
            if (tap < taps) {
                const int kh = tap / p.KW, kw = tap - kh * p.KW;
                v = load_f32(w + (int64_t)c * p.ws[0] + (int64_t)kh * p.ws[2] +
                             (int64_t)kw * p.ws[3]);
            } else if (p.has_bias) {
                v = load_f32(b + (int64_t)c * p.bs);
            }
        }
        line_w[e] = v;
    }
    __syncthreads();

    const int cvl = t % g.CVb, lane_strip = t / g.CVb;
    if (lane_strip >= g.PB) return;              // threads past the last full strip lane
    const int cv = blockIdx.y * g.CVb + cvl;
    if (cv >= g.CV) return;
    const int c0 = cv * VEC;
    const float2 *wv = reinterpret_cast<const float2 *>(line_w) + cvl * P;
    float2 bias[P];
#pragma unroll
    for (int k = 0; k < P; ++k) bias[k] = wv[(taps * cb) / 2 + k];

    for (int64_t item = (int64_t)blockIdx.x * g.PB + lane_strip; item < g.items;
         item += (int64_t)gridDim.x * g.PB) {
        const int sx = (int)(item % g.NSW);
        const int64_t r = item / g.NSW;
        const int oh = (int)(r % p.OH);
        const int n = (int)(r / p.OH);
        const int ow0 = sx * S;
        float2 acc[S][P];
#pragma unroll
        for (int i = 0; i < S; ++i)
#pragma unroll
            for (int k = 0; k < P; ++k) acc[i][k] = bias[k];
        const T *xn = x + (int64_t)n * p.xs[0] + c0;
        for (int kh = 0; kh < p.KH; ++kh) {
            const int ih = tap_input<TR>(oh, kh, p.sh, p.pbh, p.dh, p.H);
            if (ih < 0) continue;
            const T *xr = xn + (int64_t)ih * p.xs[2];
            for (int kw = 0; kw < p.KW; ++kw) {
                float2 wk[P];
                const float2 *src = wv + ((kh * p.KW + kw) * cb) / 2;
#pragma unroll
                for (int k = 0; k < P; ++k) wk[k] = src[k];
#pragma unroll
                for (int i = 0; i < S; ++i) {
                    const int iw = tap_input<TR>(ow0 + i, kw, p.sw, p.pbw, p.dw, p.W);
                    if (iw < 0 || ow0 + i >= p.OW) continue;
                    V v;
                    IO::load(v, xr + (int64_t)iw * p.xs[3]);
                    float2 xf[P];
                    widen<T, VEC>(v, xf);
#pragma unroll
                    for (int k = 0; k < P; ++k) fma2_packed(acc[i][k], wk[k], xf[k]);
                }
            }
        }
        T *yp = y + (int64_t)n * p.ys[0] + (int64_t)oh * p.ys[2] + (int64_t)ow0 * p.ys[3] + c0;
#pragma unroll
        for (int i = 0; i < S; ++i)
            if (ow0 + i < p.OW) IO::store(yp + (int64_t)i * p.ys[3], pack_pairs<T, VEC>(acc[i]));
    }
}

bool line_supports(const gconv_desc &d, const Ptrs &q) {
    if (d.Cin_g != 1 || d.Cout_g != 1) return false;        // depthwise, multiplier 1
    if (d.layout != GCONV_LAYOUT_NHWC) return false;
    const int es = dtype_size(d.dtype);
    const int vec = 16 / es;
    if (d.C_out % vec != 0) return false;
    // 16-byte vector loads and stores: aligned bases, strides in whole vectors
    if (!aligned(q.x, 16) || !aligned(q.y, 16)) return false;
    if (d.x_strides[1] != 1 || d.x_strides[0] % vec || d.x_strides[2] % vec ||
        d.x_strides[3] % vec)
        return false;
    if (d.y_strides[1] != 1 || d.y_strides[3] % vec || d.y_strides[2] % vec ||
        d.y_strides[0] % vec)
        return false;
    // weights and bias staged in shared memory
    const size_t smem = (size_t)(d.KH * d.KW + 1) * 32 * vec * sizeof(float);
    if (smem > 200 * 1024) return false;
    Params p = make_params(d);
    LineGeom g;
    return line_geometry(p, es, g) && (int64_t)p.N * p.OH < INT32_MAX &&
           (g.CV + g.CVb - 1) / g.CVb <= 65535;   // channel chunks along grid y
}

cudaError_t line_launch(const Params &p, const Ptrs &q, cudaStream_t s, int *launches) {
    *launches = 1;
    LineGeom g;
    if (!line_geometry(p, dtype_size(p.dtype), g)) return cudaErrorNotSupported;
    const int chunks = (g.CV + g.CVb - 1) / g.CVb;
    int64_t bx = (g.items + g.PB - 1) / g.PB;
    const int64_t cap = (int64_t)152 * 8 * 4 / chunks + 1;   // about 8 blocks per SM, 4 passes
    if (bx > cap) bx = cap;
    if (bx > INT32_MAX) bx = INT32_MAX;
    return GCONV_DISPATCH_DTYPE(p.dtype, T, [&] {
        constexpr int VEC = line_vec<T>();
        const size_t smem = (size_t)(p.KH * p.KW + 1) * g.CVb * VEC * sizeof(float);
        auto go = [&](auto kernel) -> cudaError_t {
            cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem);
            if (e != cudaSuccess) return e;
            e = launch_pdl(kernel, dim3((unsigned)bx, (unsigned)chunks), dim3(g.CVb * g.PB), smem,
                           s, static_cast<const T *>(q.x), static_cast<const T *>(q.w),
                           static_cast<const T *>(q.b), static_cast<T *>(q.y), p, g);
            return e != cudaSuccess ? e : cudaGetLastError();
        };
        return p.transposed ? go(line_kernel<T, true>) : go(line_kernel<T, false>);
    });
}

}  // namespace

const Schedule kDwLine = {"dw_line", line_supports, line_launch};

}  // namespace gconv
