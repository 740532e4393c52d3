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
// in shared memory as fp32 [tap][channel] and are read as broadcast vectors.
// For each kernel row, a lane first issues the loads of all KW x S input
// vectors it needs (taps outside the input are skipped), so they are in
// flight together -- the other taps' reads of a pixel hit L1, and with one
// load at a time a lane would wait a full memory latency per tap -- then
// widens each and multiplies it into fp32 accumulators with packed FMAs;
// one rounding per output at the store.  The kernel width bound KWM (4 or
// 9) is a template parameter so the load slots are registers; S = 4 pixels
// per lane for KWM = 4, 2 for KWM = 9.  Blocks are persistent (as many as
// fit at once), so the weights are staged once per block.
// Transposed calls walk strips of one column phase: outputs q*s + ph for S
// consecutive q all read tap k at input q + c(ph, k) (c from a per-block
// table of (phase, tap) offsets, none when that phase skips the tap), so a
// strip needs no division and reads consecutive inputs; the output row's
// taps come from a second table the same way.  With dilation 1 the taps of
// a phase sit s apart and their offsets one apart, so the strip's inputs
// form one register window too.
// Forward calls with stride 1 keep a register sliding window instead: the
// S + KW - 1 input vectors of a strip's row are loaded and widened once, and
// every tap reads its S vectors from the window; with dilation d a strip
// holds outputs d apart (one column phase), so its taps still slide over
// consecutive window slots.
#include "device_common.cuh"
#include "gconv_internal.h"
#include "launch.cuh"
#include "stencil_math.cuh"

namespace gconv {
namespace {

// 128-thread blocks: a lane holds ~160 registers (its loads in flight), so
// smaller blocks let three of them share an SM.
constexpr int kLineThreads = 128;
// Output pixels per lane for kernel widths up to KWM.
constexpr int line_s(int KWM) { return KWM <= 4 ? 4 : 2; }
constexpr int line_kwm(int KW) { return KW <= 4 ? 4 : 9; }

template <typename T> constexpr int line_vec() { return 16 / (int)sizeof(T); }

struct LineGeom {
    int CV;      // channel vectors in the tensor
    int CVb;     // channel vectors per block (lanes along channels)
    int PB;      // strips per block pass (lanes along pixels)
    int PH;      // column phases: stride_w (transposed), dilation_w (forward at
                 // stride 1: the window form walks one phase), else 1
    int NSW;     // strips per output row and phase
    int64_t items;   // N * OH * PH * NSW, < 2^31
    int tab_w, tab_h;   // transposed: offsets of the column / row tap tables (ints)
    int tab_p;          // transposed, dilation 1: per column phase (last tap, its offset)
    FastDiv fd_nsw, fd_ph, fd_oh, fd_sh;   // item decomposition without divisions
};

// Tap tables of a transposed call (entries per phase x tap) must fit here.
constexpr int kLineTabMax = 2048;

bool line_geometry(const Params &p, int es, LineGeom &g) {
    const int vec = 16 / es;
    if (p.C_out % vec != 0) return false;
    const int S = line_s(line_kwm(p.KW));
    g.CV = p.C_out / vec;
    const int chunks = (g.CV + 31) / 32;         // balanced chunks of <= 32 vectors
    g.CVb = (g.CV + chunks - 1) / chunks;
    g.PB = kLineThreads / g.CVb;
    // Strips of one column phase ph: outputs q*PH + ph for S consecutive q.
    g.PH = p.transposed ? p.sw : (p.sw == 1 ? p.dw : 1);
    const int Q = (p.OW + g.PH - 1) / g.PH;
    g.NSW = (Q + S - 1) / S;
    g.items = (int64_t)p.N * p.OH * g.PH * g.NSW;
    if (p.transposed &&
        ((int64_t)p.sw * p.KW > kLineTabMax || (int64_t)p.sh * p.KH > kLineTabMax))
        return false;
    const int cb = g.CVb * vec;
    g.tab_w = (p.KH * p.KW + 1) * cb;            // after the fp32 weights (same 4-byte units)
    g.tab_h = g.tab_w + (p.transposed ? p.sw * p.KW : 0);
    g.tab_p = g.tab_h + (p.transposed ? p.sh * p.KH : 0);
    g.fd_nsw = FastDiv((uint32_t)g.NSW);
    g.fd_ph = FastDiv((uint32_t)g.PH);
    g.fd_oh = FastDiv((uint32_t)p.OH);
    g.fd_sh = FastDiv((uint32_t)p.sh);
    return g.CV >= 1 && g.items <= INT32_MAX;
}

size_t line_smem(const Params &p, const LineGeom &g) {
    return (size_t)(g.tab_p + (p.transposed ? 2 * p.sw : 0)) * 4;
}

// Transposed tap table entry: for phase r (0 <= r < s) and tap k, the
// offset c with input = (o - r) / s + c for every output o = r (mod s), or
// kNoTap when no output of that phase reads tap k.
constexpr int kNoTap = -0x40000000;
__device__ __forceinline__ int tr_offset(int r, int k, int s, int pb, int d) {
    const int num = r + pb - k * d;
    return (num % s == 0) ? num / s : kNoTap;
}

// UNIT: the register-window form (forward: stride 1; transposed: dilation 1).
template <typename T, bool TR, int KWM, bool UNIT>
__global__ void __launch_bounds__(kLineThreads)
line_kernel(const T *__restrict__ x, const T *__restrict__ w, const T *__restrict__ b,
            T *__restrict__ y, Params p, LineGeom g) {
    // Let the next kernel in the stream start launching; wait for the
    // previous kernel's memory before reading global memory.
    pdl_launch_dependents();
    pdl_wait();
    constexpr int VEC = line_vec<T>();
    constexpr int P = VEC / 2;
    constexpr int S = line_s(KWM);
    using V = Vec<T, VEC>;
    using IO = VecIO<16>;
    // [KH*KW + 1][CVb * VEC] fp32 weights and bias, then (transposed) the
    // column and row tap tables.
    extern __shared__ __align__(16) float line_w[];
    int *tab_w = reinterpret_cast<int *>(line_w) + g.tab_w;
    int *tab_h = reinterpret_cast<int *>(line_w) + g.tab_h;
    int *tab_p = reinterpret_cast<int *>(line_w) + g.tab_p;

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
    if constexpr (TR) {
        for (int e = t; e < p.sw * p.KW; e += blockDim.x)
            tab_w[e] = tr_offset(e / p.KW, e % p.KW, p.sw, p.pbw, p.dw);
        for (int e = t; e < p.sh * p.KH; e += blockDim.x)
            tab_h[e] = tr_offset(e / p.KH, e % p.KH, p.sh, p.pbh, p.dh);
        // With dilation 1 the taps a column phase reads are kw_last,
        // kw_last - s, ... and their offsets c_min, c_min + 1, ...: the
        // strip's inputs form one window (phase with no tap: kw_last = -1).
        for (int ph = t; ph < p.sw; ph += blockDim.x) {
            int last = -1, cmin = 0;
            for (int kw = p.KW - 1; kw >= 0; --kw) {
                const int c = tr_offset(ph, kw, p.sw, p.pbw, 1);
                if (c != kNoTap) {
                    last = kw;
                    cmin = c;
                    break;
                }
            }
            tab_p[2 * ph] = last;
            tab_p[2 * ph + 1] = cmin;
        }
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

    const uint32_t items = (uint32_t)g.items;
    for (uint32_t item = blockIdx.x * g.PB + lane_strip; item < items;
         item += gridDim.x * g.PB) {
        // Output pixel i of the strip is column ow0 + i*ostep.
        uint32_t r, sxu;
        g.fd_nsw.divmod(item, r, sxu);
        const int sx = (int)sxu;
        int ph = 0;
        if constexpr (TR || UNIT) {
            uint32_t r2, phu;
            g.fd_ph.divmod(r, r2, phu);
            ph = (int)phu;
            r = r2;
        }
        uint32_t nu, ohu;
        g.fd_oh.divmod(r, nu, ohu);
        const int oh = (int)ohu;
        const int n = (int)nu;
        const int ostep = g.PH;
        const int q0 = sx * S;                   // first q of the strip
        const int ow0 = q0 * g.PH + ph;
        float2 acc[S][P];
#pragma unroll
        for (int i = 0; i < S; ++i)
#pragma unroll
            for (int k = 0; k < P; ++k) acc[i][k] = bias[k];
        const T *xn = x + (int64_t)n * p.xs[0] + c0;
        int qh = 0, rh = 0;
        if constexpr (TR) {
            uint32_t qhu, rhu;
            g.fd_sh.divmod((uint32_t)oh, qhu, rhu);
            qh = (int)qhu;
            rh = (int)rhu;
        }
        for (int kh = 0; kh < p.KH; ++kh) {
            int ih;
            if constexpr (TR) {
                const int c = tab_h[rh * p.KH + kh];
                ih = c == kNoTap ? -1 : qh + c;
                if (ih >= p.H) ih = -1;
            } else {
                ih = oh * p.sh - p.pbh + kh * p.dh;
                if (ih >= p.H) ih = -1;
            }
            if (ih < 0) continue;
            const T *xr = xn + (int64_t)ih * p.xs[2];
            if constexpr (TR && UNIT) {
                {
                    // The phase's j-th tap from the last (kw = kw_last - j*s)
                    // reads input q + c_min + j: a window of S + nv - 1
                    // vectors, tap j and pixel i at slot j + i.
                    constexpr int NW = S + KWM - 1;
                    const int last = tab_p[2 * ph], cmin = tab_p[2 * ph + 1];
                    const int nv = last < 0 ? 0 : (int)g.fd_ph.div((uint32_t)last) + 1;
                    float2 win[NW][P];
                    const int iw0 = q0 + cmin;
#pragma unroll
                    for (int m = 0; m < NW; ++m) {
                        const int iw = iw0 + m;
                        if (m < S + nv - 1 && iw >= 0 && iw < p.W) {
                            V v;
                            IO::load(v, xr + (int64_t)iw * p.xs[3]);
                            widen<T, VEC>(v, win[m]);
                        } else {
#pragma unroll
                            for (int k = 0; k < P; ++k) win[m][k] = make_float2(0.f, 0.f);
                        }
                    }
#pragma unroll
                    for (int j = 0; j < KWM; ++j) {
                        if (j < nv) {   // a guard, not a break: the loop stays unrolled
                            const int kw = last - j * p.sw;
                            float2 wk[P];
                            const float2 *src = wv + ((kh * p.KW + kw) * cb) / 2;
#pragma unroll
                            for (int k = 0; k < P; ++k) wk[k] = src[k];
#pragma unroll
                            for (int i = 0; i < S; ++i)
#pragma unroll
                                for (int k = 0; k < P; ++k)
                                    fma2_packed(acc[i][k], wk[k], win[j + i][k]);
                        }
                    }
                    continue;
                }
            }
            if constexpr (!TR && UNIT) {
                // Stride 1: the strip's outputs (q0 + i)*d + ph at tap kw read
                // input (q0 + i + kw)*d + ph - pb, so its S + KW - 1 input
                // vectors form one window; each is loaded and widened once
                // and slides under the taps.
                constexpr int NW = S + KWM - 1;
                float2 win[NW][P];
                const int iw0 = ow0 - p.pbw;
#pragma unroll
                for (int j = 0; j < NW; ++j) {
                    const int iw = iw0 + j * p.dw;
                    if (j < S + p.KW - 1 && iw >= 0 && iw < p.W) {
                        V v;
                        IO::load(v, xr + (int64_t)iw * p.xs[3]);
                        widen<T, VEC>(v, win[j]);
                    } else {
#pragma unroll
                        for (int k = 0; k < P; ++k) win[j][k] = make_float2(0.f, 0.f);
                    }
                }
#pragma unroll
                for (int kw = 0; kw < KWM; ++kw) {
                    if (kw >= p.KW) break;
                    float2 wk[P];
                    const float2 *src = wv + ((kh * p.KW + kw) * cb) / 2;
#pragma unroll
                    for (int k = 0; k < P; ++k) wk[k] = src[k];
#pragma unroll
                    for (int i = 0; i < S; ++i)
#pragma unroll
                        for (int k = 0; k < P; ++k) fma2_packed(acc[i][k], wk[k], win[i + kw][k]);
                }
                continue;
            }
            // Every load of this kernel row first ...
            V raw[KWM][S];
            bool ok[KWM][S];
#pragma unroll
            for (int kw = 0; kw < KWM; ++kw) {
                int base;                        // input column of pixel 0 at tap kw
                bool tap_ok = kw < p.KW;
                if constexpr (TR) {
                    const int c = tap_ok ? tab_w[ph * p.KW + kw] : kNoTap;
                    tap_ok = c != kNoTap;
                    base = q0 + c;
                } else {
                    base = ow0 * p.sw - p.pbw + kw * p.dw;
                }
#pragma unroll
                for (int i = 0; i < S; ++i) {
                    const int iw = base + i * (TR ? 1 : p.sw);
                    ok[kw][i] = tap_ok && iw >= 0 && iw < p.W && ow0 + i * ostep < p.OW;
                    if (ok[kw][i]) IO::load(raw[kw][i], xr + (int64_t)iw * p.xs[3]);
                }
            }
            // ... then the arithmetic.
#pragma unroll
            for (int kw = 0; kw < KWM; ++kw) {
                if (kw >= p.KW) break;
                float2 wk[P];
                const float2 *src = wv + ((kh * p.KW + kw) * cb) / 2;
#pragma unroll
                for (int k = 0; k < P; ++k) wk[k] = src[k];
#pragma unroll
                for (int i = 0; i < S; ++i) {
                    if (!ok[kw][i]) continue;
                    float2 xf[P];
                    widen<T, VEC>(raw[kw][i], xf);
#pragma unroll
                    for (int k = 0; k < P; ++k) fma2_packed(acc[i][k], wk[k], xf[k]);
                }
            }
        }
        T *yp = y + (int64_t)n * p.ys[0] + (int64_t)oh * p.ys[2] + (int64_t)ow0 * p.ys[3] + c0;
#pragma unroll
        for (int i = 0; i < S; ++i)
            if (ow0 + i * ostep < p.OW)
                IO::store(yp + (int64_t)i * ostep * p.ys[3], pack_pairs<T, VEC>(acc[i]));
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
    Params p = make_params(d);
    LineGeom g;
    if (!line_geometry(p, es, g)) return false;
    // weights, bias and tap tables in shared memory
    if (line_smem(p, g) > 200 * 1024) return false;
    return (int64_t)p.N * p.OH < INT32_MAX &&
           (g.CV + g.CVb - 1) / g.CVb <= 65535;   // channel chunks along grid y
}

cudaError_t line_launch(const Params &p, const Ptrs &q, cudaStream_t s, int *launches) {
    *launches = 1;
    LineGeom g;
    if (!line_geometry(p, dtype_size(p.dtype), g)) return cudaErrorNotSupported;
    const int chunks = (g.CV + g.CVb - 1) / g.CVb;
    const size_t smem = line_smem(p, g);
    return GCONV_DISPATCH_DTYPE(p.dtype, T, [&] {
        auto go = [&](auto kernel) -> cudaError_t {
            cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem);
            if (e != cudaSuccess) return e;
            // Persistent blocks: as many as fit on the GPU at once, so the
            // weight staging happens once per block; strips are grid-strided.
            int per_sm = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel,
                                                              g.CVb * g.PB, smem);
            if (e != cudaSuccess) return e;
            if (per_sm < 1) per_sm = 1;
            int64_t bx = (int64_t)152 * per_sm / chunks;
            if (bx < 1) bx = 1;
            const int64_t need = (g.items + g.PB - 1) / g.PB;
            if (bx > need) bx = need;
            if (bx > INT32_MAX) bx = INT32_MAX;
            e = launch_kernel(kernel, dim3((unsigned)bx, (unsigned)chunks), dim3(g.CVb * g.PB), smem,
                           s, static_cast<const T *>(q.x), static_cast<const T *>(q.w),
                           static_cast<const T *>(q.b), static_cast<T *>(q.y), p, g);
            return e != cudaSuccess ? e : cudaGetLastError();
        };
        // The window forms: forward with stride 1 (one column phase per
        // strip when dilated), transposed with dilation 1.
        const bool win = p.transposed ? p.dw == 1 : p.sw == 1;
        if (line_kwm(p.KW) == 4) {
            if (p.transposed)
                return win ? go(line_kernel<T, true, 4, true>) : go(line_kernel<T, true, 4, false>);
            return win ? go(line_kernel<T, false, 4, true>) : go(line_kernel<T, false, 4, false>);
        }
        if (p.transposed)
            return win ? go(line_kernel<T, true, 9, true>) : go(line_kernel<T, true, 9, false>);
        return win ? go(line_kernel<T, false, 9, true>) : go(line_kernel<T, false, 9, false>);
    });
}

}  // namespace

const Schedule kDwLine = {"dw_line", line_supports, line_launch};

}  // namespace gconv
