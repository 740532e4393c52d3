// k_wgrad.cu -- the backward pass for the weight and the bias:
//   dw[co, ci, kh, kw] = sum_{n, oh, ow} gy[n, co, oh, ow] * x[n, g*Cin_g + ci, ih, iw]
//   db[co]             = sum_{n, oh, ow} gy[n, co, oh, ow]
// with (ih, iw) the forward taps (torch/_inductor/kernel/conv.py,
// convolution_backward_lowering: grad weight, and grad bias as the sum of
// grad_output over batch and space).
//
// Two launches.  The first splits the output pixels (n, oh, ow) into slices
// and writes one fp32 partial sum per (slice, co, tap) -- bias as one more
// tap -- into the caller's workspace [slice][C_out][Cin_g*KH*KW + 1]; the
// second adds each entry's slices (compensated fp32, as accurate as twice
// the precision) in a fixed order (32 interleaved runs of slices, then a
// fixed tree over the run sums) and rounds once into dw (dense
// [C_out, Cin_g, KH, KW]) and db.  No atomics: the result is the same on
// every run.
//
// Partial pass, four forms:
//  - channels-last depthwise 3x3 at square stride 1 or 2 (dilation 1): the
//    forward's TMA row ring with x and gy rows staged together
//    (k_wgrad_row.cu);
//  - channels-last depthwise (one input and one output channel per group):
//    a block owns a chunk of channel vectors and a slice of pixels; lane
//    (cv, pixel lane) keeps CH channels x every tap in fp32 registers, walks
//    its pixels (for each: the gy vector and the x vector of every tap in the
//    input are loaded first, so they are in flight together, then packed
//    FMAs), and the block adds its pixel lanes in shared memory, one tap at a
//    time in a fixed order;
//  - the same with kernels of at most 3 x 3 (or 1 x 9) at column stride 1
//    (any dilation) or 2 (dilation 1): strips of 4 outputs that share one
//    register window of inputs per kernel row (wgrad_strip_kernel);
//  - any other layout or group shape: a block owns (slice, co), every thread
//    sums a tap over its pixels through the strides, and a fixed-order block
//    reduction (shuffles, then shared memory) gives the slice's value.
#include "device_common.cuh"
#include "gconv_internal.h"
#include "launch.cuh"
#include "stencil_math.cuh"

namespace gconv {
namespace {

constexpr int kWgThreads = 256;
constexpr int kWgBlocksTarget = 152 * 2;   // measured: 4 and 8 per SM are slower (more slices to add)

// Channels per lane for the channels-last form: all taps of CH channels in
// fp32 registers, plus one load slot per tap.
template <typename T, int TMAX> constexpr int wg_ch() { return TMAX <= 9 ? 4 : 2; }

struct WgPlan {
    bool cl;          // channels-last depthwise form
    int tmax;         // 9, 25 or 49 (cl form)
    int ch;           // channels per lane (cl form)
    int CVb, PL;      // lanes along channels / pixels (cl form)
    int chunks;       // channel chunks (cl form)
    int slices;
    int64_t P;        // output pixels N * OH * OW
    int T1;           // Cin_g * KH * KW + 1
    FastDiv fd_ow, fd_oh;   // pixel index -> (n, oh, ow) when P < 2^32
    // strip form: items (n, oh, column phase, strip of kWgS outputs)
    int strip;        // 0: per-pixel form; 33 or 19: strip form for KH<=3,KW<=3 / KH=1,KW<=9
                      // at column stride 1; 233 or 219: the same at column stride 2
    int PH, NSW;
    int64_t items;
    FastDiv fd_nsw, fd_ph;
};

constexpr int kWgS = 4;   // output pixels per strip (strip form)

// Output pixel q -> (n, oh, ow): multiply-high divisions when q fits in 32
// bits (always, short of 2^32 pixels), 64-bit divisions otherwise.
__device__ __forceinline__ void pixel_of(int64_t q, const Params &p, const WgPlan &pl, int &n,
                                         int &oh, int &ow) {
    if (pl.P <= (int64_t)0xFFFFFFFFu) {
        uint32_t r, owu, nu, ohu;
        pl.fd_ow.divmod((uint32_t)q, r, owu);
        pl.fd_oh.divmod(r, nu, ohu);
        n = (int)nu; oh = (int)ohu; ow = (int)owu;
    } else {
        ow = (int)(q % p.OW);
        const int64_t r = q / p.OW;
        oh = (int)(r % p.OH);
        n = (int)(r / p.OH);
    }
}

int cl_tmax(const Params &p) {
    const int taps = p.KH * p.KW;
    return taps <= 9 ? 9 : (taps <= 25 ? 25 : (taps <= 49 ? 49 : 0));
}

int cl_ch(const Params &p, int tmax) {
    (void)p;
    return tmax <= 9 ? 4 : 2;
}

// The shape half of the channels-last test (the pointer half is in
// wg_cl_pointers); the workspace size depends on the shape only.
bool cl_shape(const Params &p) {
    if (p.Cin_g != 1 || p.Cout_g != 1 || p.layout != GCONV_LAYOUT_NHWC) return false;
    const int tmax = cl_tmax(p);
    if (!tmax) return false;
    const int ch = cl_ch(p, tmax);
    if (p.C_out % ch) return false;
    if (p.xs[1] != 1 || p.xs[0] % ch || p.xs[2] % ch || p.xs[3] % ch) return false;
    if (p.ys[1] != 1 || p.ys[0] % ch || p.ys[2] % ch || p.ys[3] % ch) return false;
    return (int64_t)p.C_out / ch / 32 < 65535;   // channel chunks along grid y
}

bool wg_cl_pointers(const Params &p, const void *x, const void *gy, int ch) {
    const uintptr_t a = (uintptr_t)(ch * dtype_size(p.dtype));
    return aligned(x, a) && aligned(gy, a);
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The strip form takes channels-last depthwise calls with kernels of at most
// 3 x 3, or height 1 and width at most 9, at column stride 1 (any dilation)
// or column stride 2 (column dilation 1).
int strip_kind(const Params &p) {
    if (!cl_shape(p)) return 0;
    int base = 0;
    if (p.KH <= 3 && p.KW <= 3) base = 33;
    else if (p.KH == 1 && p.KW <= 9) base = 19;
    if (!base) return 0;
    if (p.sw == 1) return base;
    if (p.sw == 2 && p.dw == 1) return 200 + base;   // stride 2: window of contiguous columns
    return 0;
}

WgPlan plan_for(const Params &p, bool cl, int strip = 0) {
    WgPlan w{};
    w.P = (int64_t)p.N * p.OH * p.OW;
    w.T1 = p.Cin_g * p.KH * p.KW + 1;
    w.cl = cl;
    w.fd_ow = FastDiv((uint32_t)(p.OW > 0 ? p.OW : 1));
    w.fd_oh = FastDiv((uint32_t)(p.OH > 0 ? p.OH : 1));
    if (strip) {
        // 4 channels a lane; strips of kWgS outputs of one column phase.
        w.strip = strip;
        w.ch = 4;
        const int cv = p.C_out / w.ch;
        w.chunks = (int)cdiv(cv, 32);
        w.CVb = (int)cdiv(cv, w.chunks);
        w.PL = kWgThreads / w.CVb;
        w.PH = strip > 200 ? 1 : p.dw;
        const int Q = (p.OW + w.PH - 1) / w.PH;
        w.NSW = (Q + kWgS - 1) / kWgS;
        w.items = (int64_t)p.N * p.OH * w.PH * w.NSW;
        w.fd_nsw = FastDiv((uint32_t)w.NSW);
        w.fd_ph = FastDiv((uint32_t)w.PH);
        int64_t s = cdiv(kWgBlocksTarget, w.chunks);
        const int64_t most = cdiv(w.items, (int64_t)w.PL * 2);   // at least ~2 strips per lane
        if (s > most) s = most;
        w.slices = (int)(s < 1 ? 1 : s);
    } else if (cl) {
        w.tmax = cl_tmax(p);
        w.ch = cl_ch(p, w.tmax);
        // Chunks of at most 32 channel vectors, balanced (36 vectors: 2 x 18).
        const int cv = p.C_out / w.ch;
        w.chunks = (int)cdiv(cv, 32);
        w.CVb = (int)cdiv(cv, w.chunks);
        w.PL = kWgThreads / w.CVb;
        int64_t s = cdiv(kWgBlocksTarget, w.chunks);
        const int64_t most = cdiv(w.P, (int64_t)w.PL * 4);   // at least ~4 pixels per lane
        if (s > most) s = most;
        w.slices = (int)(s < 1 ? 1 : s);
    } else {
        int64_t s = cdiv(kWgBlocksTarget, p.C_out > 0 ? p.C_out : 1);
        const int64_t most = cdiv(w.P, kWgThreads);
        if (s > most) s = most;
        w.slices = (int)(s < 1 ? 1 : s);
    }
    return w;
}

// Pixel range [p0, p1) of slice `sl`.
__device__ __forceinline__ void slice_range(int64_t P, int slices, int sl, int64_t &p0,
                                            int64_t &p1) {
    const int64_t per = P / slices, extra = P % slices;
    p0 = sl * per + (sl < extra ? sl : extra);
    p1 = p0 + per + (sl < extra ? 1 : 0);
}

template <typename T, int TMAX, int CH>
__global__ void __launch_bounds__(kWgThreads)
wgrad_cl_kernel(const T *__restrict__ x, const T *__restrict__ gy, float *__restrict__ ws,
                Params p, WgPlan pl) {
    pdl_launch_dependents();
    pdl_wait();
    constexpr int PR = CH / 2;                    // channel pairs
    using V = Vec<T, CH>;
    using IO = VecIO<CH * (int)sizeof(T)>;
    __shared__ float red[kWgThreads * CH];        // [pixel lane][block channel]

    const int t = threadIdx.x;
    const int cvl = t % pl.CVb, lp = t / pl.CVb;
    const int cv = blockIdx.y * pl.CVb + cvl;
    const bool active = lp < pl.PL && cv * CH < p.C_out;
    const int c0 = cv * CH;
    const int taps = p.KH * p.KW;
    int64_t p0, p1;
    slice_range(pl.P, pl.slices, blockIdx.x, p0, p1);

    float2 acc[TMAX][PR];
    float2 accb[PR];
#pragma unroll
    for (int k = 0; k < PR; ++k) accb[k] = make_float2(0.f, 0.f);
#pragma unroll
    for (int tp = 0; tp < TMAX; ++tp)
#pragma unroll
        for (int k = 0; k < PR; ++k) acc[tp][k] = make_float2(0.f, 0.f);

    if (active) {
        // U pixels per step (q, q + PL, ...; two for kernels of up to 9
        // taps), their loads all issued before any arithmetic: gy and the x
        // vector of every tap in the input.
        constexpr int U = TMAX <= 9 ? 2 : 1;
        for (int64_t q = p0 + lp; q < p1; q += U * pl.PL) {
            V gv[U];
            V xv[U][TMAX];
            bool ok[U][TMAX];
            bool have[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t qu = q + u * pl.PL;
                have[u] = qu < p1;
                int n, oh, ow;
                pixel_of(have[u] ? qu : p0, p, pl, n, oh, ow);
                if (have[u])
                    IO::load(gv[u], gy + (int64_t)n * p.ys[0] + (int64_t)oh * p.ys[2] +
                                        (int64_t)ow * p.ys[3] + c0);
                const T *xn = x + (int64_t)n * p.xs[0] + c0;
                const int ih0 = oh * p.sh - p.pbh, iw0 = ow * p.sw - p.pbw;
                int kh = 0, kw = 0;   // tap tp = kh*KW + kw, stepped without divisions
#pragma unroll
                for (int tp = 0; tp < TMAX; ++tp) {
                    ok[u][tp] = false;
                    if (have[u] && tp < taps) {
                        const int ih = ih0 + kh * p.dh, iw = iw0 + kw * p.dw;
                        ok[u][tp] = ih >= 0 && ih < p.H && iw >= 0 && iw < p.W;
                        if (ok[u][tp])
                            IO::load(xv[u][tp], xn + (int64_t)ih * p.xs[2] + (int64_t)iw * p.xs[3]);
                    }
                    if (++kw == p.KW) {
                        kw = 0;
                        ++kh;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (!have[u]) continue;
                float2 g2[PR];
                widen<T, CH>(gv[u], g2);
#pragma unroll
                for (int k = 0; k < PR; ++k) {
                    accb[k].x += g2[k].x;
                    accb[k].y += g2[k].y;
                }
#pragma unroll
                for (int tp = 0; tp < TMAX; ++tp) {
                    if (ok[u][tp]) {
                        float2 x2[PR];
                        widen<T, CH>(xv[u][tp], x2);
#pragma unroll
                        for (int k = 0; k < PR; ++k) fma2_packed(acc[tp][k], g2[k], x2[k]);
                    }
                }
            }
        }
    }
    // Add the pixel lanes, one tap (then the bias) at a time, lanes in order.
    const int cb = pl.CVb * CH;
    const int c_first = blockIdx.y * cb;
#pragma unroll
    for (int tp = 0; tp <= TMAX; ++tp) {
        const bool bias_slot = tp == TMAX;
        if (!bias_slot && tp >= taps) continue;   // the same for the whole block
        const float2 *src = bias_slot ? accb : acc[bias_slot ? 0 : tp];
        const int slot = bias_slot ? taps : tp;
        if (lp < pl.PL) {
#pragma unroll
            for (int k = 0; k < PR; ++k) {
                red[lp * cb + cvl * CH + 2 * k] = src[k].x;
                red[lp * cb + cvl * CH + 2 * k + 1] = src[k].y;
            }
        }
        __syncthreads();
        for (int e = t; e < cb; e += blockDim.x) {
            const int c = c_first + e;
            if (c < p.C_out) {
                float s = 0.f;
                for (int l = 0; l < pl.PL; ++l) s += red[l * cb + e];
                ws[((int64_t)blockIdx.x * p.C_out + c) * pl.T1 + slot] = s;
            }
        }
        __syncthreads();
    }
}

template <typename T>
__global__ void __launch_bounds__(kWgThreads)
wgrad_generic_kernel(const T *__restrict__ x, const T *__restrict__ gy, float *__restrict__ ws,
                     Params p, WgPlan pl) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ float warp_sums[kWgThreads / 32];
    const int t = threadIdx.x;
    const int khw = p.KH * p.KW;
    int64_t p0, p1;
    slice_range(pl.P, pl.slices, blockIdx.x, p0, p1);
    for (int co = blockIdx.y; co < p.C_out; co += gridDim.y) {
        const int g = co / p.Cout_g;
        for (int tap = 0; tap < pl.T1; ++tap) {
            const bool is_bias = tap == pl.T1 - 1;
            const int ci = is_bias ? 0 : tap / khw;
            const int k = is_bias ? 0 : tap - ci * khw;
            const int kh = k / p.KW, kw = k - kh * p.KW;
            const T *xc = x + (int64_t)(g * p.Cin_g + ci) * p.xs[1];
            float s = 0.f;
            for (int64_t q = p0 + t; q < p1; q += blockDim.x) {
                int n, oh, ow;
                pixel_of(q, p, pl, n, oh, ow);
                const float gv = load_f32(gy + (int64_t)n * p.ys[0] + (int64_t)co * p.ys[1] +
                                          (int64_t)oh * p.ys[2] + (int64_t)ow * p.ys[3]);
                if (is_bias) {
                    s += gv;
                } else {
                    const int ih = tap_input<false>(oh, kh, p.sh, p.pbh, p.dh, p.H);
                    const int iw = tap_input<false>(ow, kw, p.sw, p.pbw, p.dw, p.W);
                    if (ih >= 0 && iw >= 0)
                        s = fmaf(gv, load_f32(xc + (int64_t)n * p.xs[0] + (int64_t)ih * p.xs[2] +
                                              (int64_t)iw * p.xs[3]),
                                 s);
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
            if (t % 32 == 0) warp_sums[t / 32] = s;
            __syncthreads();
            if (t == 0) {
                float tot = 0.f;
                for (int i = 0; i < kWgThreads / 32; ++i) tot += warp_sums[i];
                ws[((int64_t)blockIdx.x * p.C_out + co) * pl.T1 + tap] = tot;
            }
            __syncthreads();
        }
    }
}

// Strip form of the partial pass: lane (cv, strip lane) walks items
// (n, oh, column phase ph, strip of kWgS outputs ow = (q0 + i)*d + ph).  Per
// item it loads the strip's gy vectors once, and for each kernel row the
// strip's window of input vectors: at column stride 1, kWgS + KW - 1 of them
// d apart (output i at tap kw reads slot i + kw); at column stride 2 (SW = 2,
// dilation 1, one phase), 2*(kWgS - 1) + KW contiguous ones (output i at tap
// kw reads slot 2i + kw).  A pixel then costs 1 + KH*(window)/kWgS vector
// loads instead of 1 + KH*KW, all of a row in flight together.
template <typename T, int KHM, int KWM, int SW>
__global__ void __launch_bounds__(kWgThreads)
wgrad_strip_kernel(const T *__restrict__ x, const T *__restrict__ gy, float *__restrict__ ws,
                   Params p, WgPlan pl) {
    pdl_launch_dependents();
    pdl_wait();
    constexpr int CH = 4;
    constexpr int PR = CH / 2;
    constexpr int S = kWgS;
    constexpr int NW = (S - 1) * SW + KWM;
    using V = Vec<T, CH>;
    using IO = VecIO<CH * (int)sizeof(T)>;
    __shared__ float red[kWgThreads * CH];        // [pixel lane][block channel]
    const int nw = (S - 1) * SW + p.KW;           // window slots in use
    const int jstep = SW == 1 ? p.dw : 1;         // columns between slots

    const int t = threadIdx.x;
    const int cvl = t % pl.CVb, lp = t / pl.CVb;
    const int cv = blockIdx.y * pl.CVb + cvl;
    const bool active = lp < pl.PL && cv * CH < p.C_out;
    const int c0 = cv * CH;
    int64_t i0, i1;
    slice_range(pl.items, pl.slices, blockIdx.x, i0, i1);

    float2 acc[KHM][KWM][PR];
    float2 accb[PR];
#pragma unroll
    for (int k = 0; k < PR; ++k) accb[k] = make_float2(0.f, 0.f);
#pragma unroll
    for (int a = 0; a < KHM; ++a)
#pragma unroll
        for (int c = 0; c < KWM; ++c)
#pragma unroll
            for (int k = 0; k < PR; ++k) acc[a][c][k] = make_float2(0.f, 0.f);

    if (active) {
        for (int64_t item = i0 + lp; item < i1; item += pl.PL) {
            uint32_t r, sxu, r2, phu, nu, ohu;
            pl.fd_nsw.divmod((uint32_t)item, r, sxu);
            pl.fd_ph.divmod(r, r2, phu);
            pl.fd_oh.divmod(r2, nu, ohu);
            const int oh = (int)ohu, n = (int)nu;
            const int ow0 = (int)sxu * S * pl.PH + (int)phu;
            float2 g[S][PR];
#pragma unroll
            for (int i = 0; i < S; ++i) {
                const int ow = ow0 + i * pl.PH;
                if (ow < p.OW) {
                    V v;
                    IO::load(v, gy + (int64_t)n * p.ys[0] + (int64_t)oh * p.ys[2] +
                                    (int64_t)ow * p.ys[3] + c0);
                    widen<T, CH>(v, g[i]);
                } else {
#pragma unroll
                    for (int k = 0; k < PR; ++k) g[i][k] = make_float2(0.f, 0.f);
                }
#pragma unroll
                for (int k = 0; k < PR; ++k) {
                    accb[k].x += g[i][k].x;
                    accb[k].y += g[i][k].y;
                }
            }
            const T *xn = x + (int64_t)n * p.xs[0] + c0;
            const int iw0 = ow0 * SW - p.pbw;
#pragma unroll
            for (int kh = 0; kh < KHM; ++kh) {
                const int ih = oh * p.sh - p.pbh + kh * p.dh;
                if (kh >= p.KH || ih < 0 || ih >= p.H) continue;   // guards keep it unrolled
                const T *xr = xn + (int64_t)ih * p.xs[2];
                float2 win[NW][PR];
#pragma unroll
                for (int j = 0; j < NW; ++j) {
                    const int iw = iw0 + j * jstep;
                    if (j < nw && iw >= 0 && iw < p.W) {
                        V v;
                        IO::load(v, xr + (int64_t)iw * p.xs[3]);
                        widen<T, CH>(v, win[j]);
                    } else {
#pragma unroll
                        for (int k = 0; k < PR; ++k) win[j][k] = make_float2(0.f, 0.f);
                    }
                }
#pragma unroll
                for (int kw = 0; kw < KWM; ++kw) {
                    if (kw < p.KW) {
#pragma unroll
                        for (int i = 0; i < S; ++i)
#pragma unroll
                            for (int k = 0; k < PR; ++k)
                                fma2_packed(acc[kh][kw][k], g[i][k], win[i * SW + kw][k]);
                    }
                }
            }
        }
    }
    // Add the pixel lanes, one tap (then the bias) at a time, lanes in order.
    const int cb = pl.CVb * CH;
    const int c_first = blockIdx.y * cb;
#pragma unroll
    for (int tp = 0; tp <= KHM * KWM; ++tp) {
        const bool bias_slot = tp == KHM * KWM;
        const int kh = bias_slot ? 0 : tp / KWM, kw = bias_slot ? 0 : tp % KWM;
        if (!bias_slot && (kh >= p.KH || kw >= p.KW)) continue;   // the same for the block
        const float2 *src = bias_slot ? accb : acc[kh][kw];
        const int slot = bias_slot ? p.KH * p.KW : kh * p.KW + kw;
        if (lp < pl.PL) {
#pragma unroll
            for (int k = 0; k < PR; ++k) {
                red[lp * cb + cvl * CH + 2 * k] = src[k].x;
                red[lp * cb + cvl * CH + 2 * k + 1] = src[k].y;
            }
        }
        __syncthreads();
        for (int e = t; e < cb; e += blockDim.x) {
            const int c = c_first + e;
            if (c < p.C_out) {
                float sum = 0.f;
                for (int l = 0; l < pl.PL; ++l) sum += red[l * cb + e];
                ws[((int64_t)blockIdx.x * p.C_out + c) * pl.T1 + slot] = sum;
            }
        }
        __syncthreads();
    }
}

// Second pass: entry e = (co, tap) of the [C_out][T1] table is the sum of
// its slices.  A block owns 8 consecutive entries (one 32-byte sector per
// slice) and its 32 groups take slices g, g+32, g+64, ... (four loads in
// flight at a time), each adding them in slice order; the 32 group sums are
// then added pairwise in a fixed tree.  The order is fixed, so the result is
// the same on every run.
//
// The sums are compensated fp32 (a rounded sum plus its running error): each
// addition is Knuth's error-free TwoSum and the errors are added up, as in
// the cascaded summation of Ogita, Rump and Oishi, "Accurate sum and dot
// product" (SIAM J. Sci. Comput., 2005), which is as accurate as summing in
// twice the precision and rounding once.  FP64 would give the same accuracy,
// but its pipe on this GPU is far slower than the FP32 pipes.  The explicit
// round-to-nearest intrinsics keep the compiler from merging or reordering
// the additions.
constexpr int kFinEntries = 8, kFinGroups = 32;

struct Sum2 {
    float hi, lo;
};

__device__ __forceinline__ void two_sum_add(Sum2 &acc, float v) {
    const float s = __fadd_rn(acc.hi, v);
    const float bb = __fsub_rn(s, acc.hi);
    const float err = __fadd_rn(__fsub_rn(acc.hi, __fsub_rn(s, bb)), __fsub_rn(v, bb));
    acc.hi = s;
    acc.lo = __fadd_rn(acc.lo, err);
}

__device__ __forceinline__ void two_sum_merge(Sum2 &acc, const Sum2 &o) {
    const float lo = __fadd_rn(acc.lo, o.lo);
    two_sum_add(acc, o.hi);
    acc.lo = __fadd_rn(acc.lo, lo);
}

template <typename T>
__global__ void __launch_bounds__(kFinEntries * kFinGroups)
wgrad_finish_kernel(const float *__restrict__ ws, T *__restrict__ dw, T *__restrict__ db,
                    int C_out, int T1, int slices) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ Sum2 part[kFinGroups][kFinEntries];
    const int lane = threadIdx.x % kFinEntries, grp = threadIdx.x / kFinEntries;
    const int64_t total = (int64_t)C_out * T1;
    const int64_t e = (int64_t)blockIdx.x * kFinEntries + lane;
    Sum2 s{0.f, 0.f};
    if (e < total) {
        int sl = grp;
        for (; sl + 3 * kFinGroups < slices; sl += 4 * kFinGroups) {
            const float a = ws[(int64_t)sl * total + e];
            const float b = ws[(int64_t)(sl + kFinGroups) * total + e];
            const float c = ws[(int64_t)(sl + 2 * kFinGroups) * total + e];
            const float d = ws[(int64_t)(sl + 3 * kFinGroups) * total + e];
            two_sum_add(s, a);
            two_sum_add(s, b);
            two_sum_add(s, c);
            two_sum_add(s, d);
        }
        for (; sl < slices; sl += kFinGroups) two_sum_add(s, ws[(int64_t)sl * total + e]);
    }
    part[grp][lane] = s;
    __syncthreads();
#pragma unroll
    for (int h = kFinGroups / 2; h >= 1; h /= 2) {
        if (grp < h) {
            Sum2 m = part[grp][lane];
            two_sum_merge(m, part[grp + h][lane]);
            part[grp][lane] = m;
        }
        __syncthreads();
    }
    if (grp == 0 && e < total) {
        const Sum2 tot = part[0][lane];
        // An infinite sum leaves a NaN error term behind: keep the infinity.
        const float v = isinf(tot.hi) ? tot.hi : __fadd_rn(tot.hi, tot.lo);
        const int co = (int)(e / T1), tap = (int)(e - (int64_t)co * T1);
        if (tap < T1 - 1)
            dw[(int64_t)co * (T1 - 1) + tap] = from_f32<T>(v);
        else if (db)
            db[co] = from_f32<T>(v);
    }
}

template <typename T, int TMAX>
cudaError_t launch_cl(const Params &p, const T *x, const T *gy, float *ws, const WgPlan &pl,
                      cudaStream_t s) {
    constexpr int CH = wg_ch<T, TMAX>();
    return launch_kernel(wgrad_cl_kernel<T, TMAX, CH>, dim3(pl.slices, pl.chunks),
                      dim3(pl.CVb * pl.PL), 0, s, x, gy, ws, p, pl);
}

// The finish pass over `slices` partial slices of T1 entries per channel.
cudaError_t finish_launch(const Params &p, const float *ws, void *dw, void *db, int T1,
                          int slices, cudaStream_t s) {
    const int64_t total = (int64_t)p.C_out * T1;
    const int64_t blocks = (total + kFinEntries - 1) / kFinEntries;
    if (blocks > INT32_MAX) return cudaErrorInvalidValue;
    return GCONV_DISPATCH_DTYPE(p.dtype, T, [&] {
        cudaError_t e = launch_kernel(wgrad_finish_kernel<T>, dim3((unsigned)blocks),
                                   dim3(kFinEntries * kFinGroups), 0, s, ws,
                                   static_cast<T *>(dw), static_cast<T *>(db), p.C_out, T1, slices);
        return e != cudaSuccess ? e : cudaGetLastError();
    });
}

}  // namespace

uint64_t wgrad_workspace_bytes(const Params &p) {
    // Enough for either form, so the size does not depend on the pointers.
    const WgPlan g = plan_for(p, false);
    int slices = g.slices;
    if (cl_shape(p)) {
        const WgPlan c = plan_for(p, true);
        if (c.slices > slices) slices = c.slices;
        const int sk = strip_kind(p);
        if (sk && (int64_t)p.N * p.OH * p.OW < 0xFFFFFFFFll) {
            const WgPlan st = plan_for(p, true, sk);
            if (st.slices > slices) slices = st.slices;
        }
    }
    const int rs = wgrad_row_slices(p);
    if (rs > slices) slices = rs;
    uint64_t b = (uint64_t)slices * (uint64_t)(p.C_out > 0 ? p.C_out : 0) * (uint64_t)g.T1 * 4u;
    return b < 16 ? 16 : b;
}

cudaError_t wgrad_launch(const Params &p, const void *x, const void *gy, void *dw, void *db,
                         void *workspace, cudaStream_t s, int *launches) {
    *launches = 2;
    float *ws = static_cast<float *>(workspace);
    const int rs = wgrad_row_slices(p);
    if (rs && wgrad_row_pointers(x, gy)) {
        // Depthwise 3x3 on the row ring, then the same finish.
        cudaError_t e = wgrad_row_partial(p, x, gy, ws, s);
        if (e != cudaSuccess) return e;
        return finish_launch(p, ws, dw, db, p.KH * p.KW + 1, rs, s);
    }
    bool cl = cl_shape(p);
    if (cl) cl = wg_cl_pointers(p, x, gy, cl_ch(p, cl_tmax(p)));
    // The strip form (4-channel loads, items counted in 32 bits).
    int sk = cl ? strip_kind(p) : 0;
    if (sk && !(wg_cl_pointers(p, x, gy, 4) && (int64_t)p.N * p.OH * p.OW < 0xFFFFFFFFll))
        sk = 0;
    const WgPlan pl = plan_for(p, cl, sk);
    return GCONV_DISPATCH_DTYPE(p.dtype, T, [&] {
        const T *xt = static_cast<const T *>(x);
        const T *gt = static_cast<const T *>(gy);
        cudaError_t e;
        const dim3 sg(pl.slices, pl.chunks), sb(pl.CVb * pl.PL);
        if (sk == 33) {
            e = launch_kernel(wgrad_strip_kernel<T, 3, 3, 1>, sg, sb, 0, s, xt, gt, ws, p, pl);
        } else if (sk == 19) {
            e = launch_kernel(wgrad_strip_kernel<T, 1, 9, 1>, sg, sb, 0, s, xt, gt, ws, p, pl);
        } else if (sk == 233) {
            e = launch_kernel(wgrad_strip_kernel<T, 3, 3, 2>, sg, sb, 0, s, xt, gt, ws, p, pl);
        } else if (sk == 219) {
            e = launch_kernel(wgrad_strip_kernel<T, 1, 9, 2>, sg, sb, 0, s, xt, gt, ws, p, pl);
        } else if (cl) {
            if (pl.tmax == 9) e = launch_cl<T, 9>(p, xt, gt, ws, pl, s);
            else if (pl.tmax == 25) e = launch_cl<T, 25>(p, xt, gt, ws, pl, s);
            else e = launch_cl<T, 49>(p, xt, gt, ws, pl, s);
        } else {
            const int gy_blocks = p.C_out < 65535 ? p.C_out : 65535;
            e = launch_kernel(wgrad_generic_kernel<T>, dim3(pl.slices, gy_blocks), dim3(kWgThreads), 0,
                           s, xt, gt, ws, p, pl);
        }
        if (e != cudaSuccess) return e;
        return finish_launch(p, ws, dw, db, pl.T1, pl.slices, s);
    });
}

}  // namespace gconv
