// k_mult.cu -- dw_mult: depthwise convolution with a channel multiplier
// m <= 16 on NCHW input, every output channel of an input channel computed
// from one load of that input channel (executorch PR #25085, description,
// second paragraph: "all output channels of an input channel per load, for
// multipliers up to 16").
//
// Design for sm_103a:
//  - Work items are (input channel c, image n, band of BR output rows,
//    column chunk); consecutive items share c, so a persistent CTA reloads
//    the m*KH*KW weights only when c changes.  Items are split evenly over
//    two CTAs per SM.
//  - The item's input band ((BR-1)*SH + KH rows x Win columns, zero outside
//    the image) is fetched with 16-byte loads into registers one item ahead,
//    then widened once to fp32 into shared memory, placed so that every
//    thread's window starts on a 16-byte boundary.
//  - Thread (row, pixel group) computes S consecutive output pixels of one
//    output row for MB output channels at a time: per kernel row it loads
//    its (S-1)*SW + KW window with 16-byte shared loads, and per tap one
//    broadcast shared load of MB weights feeds MB*S FMAs.  Kernel widths up
//    to 9 are handled by a fully unrolled, predicated tap loop.
//  - fp32 accumulation from the bias, one rounding, 16-byte stores of S
//    pixels where the row allows it.
#include "device_common.cuh"
#include "gconv_internal.h"

namespace gconv {
namespace {

constexpr int kMultThreads = 256;
constexpr int kMultMaxChunks = 4;    // 16-byte global chunks per thread per band
constexpr int kMultMaxKW = 9;

struct MultGeom {
    int m;          // multiplier (Cout_g)
    int S;          // output pixels per thread
    int PGn;        // pixel groups per row chunk
    int BR;         // output rows per band
    int OWc, CC;    // output columns per chunk, column chunks
    int bands;
    int rows_in;    // input rows per band
    int Win;        // input columns per band (window span of the chunk)
    int pitch;      // fp32 elements per shared row (multiple of 4)
    int cpr;        // 16-byte global chunks per band row
    int nchunks;    // chunks per band
    int items;
    int ctas;
    int vec_store;  // rows of y allow 16-byte stores of S pixels
};

template <typename T> struct Chunk16 {
    static constexpr int kElems = 16 / sizeof(T);
};

template <typename T, int SW, int MB, int S>
__global__ void __launch_bounds__(kMultThreads, 2)
mult_kernel(const T *__restrict__ x, const T *__restrict__ w, const T *__restrict__ b,
            T *__restrict__ y, Params p, MultGeom g) {
    constexpr int CE = Chunk16<T>::kElems;            // elements per 16-byte chunk
    constexpr int WIN = (S - 1) * SW + kMultMaxKW;    // window incl. unused taps
    constexpr int WIN4 = (WIN + 3) / 4;               // 16-byte shared loads
    extern __shared__ __align__(16) float mult_smem[];
    float *band = mult_smem;                          // rows_in x pitch
    float *wsm = band + g.rows_in * g.pitch;          // [kh][kw][m]
    float *bsm = wsm + p.KH * p.KW * g.m;             // [m]

    const int t = threadIdx.x;
    const int per = g.items / g.ctas, extra = g.items % g.ctas;
    const int i0 = blockIdx.x * per + min((int)blockIdx.x, extra);
    const int i1 = i0 + per + ((int)blockIdx.x < extra ? 1 : 0);
    if (i0 >= i1) return;

    const int row = t / g.PGn, pg = t - (t / g.PGn) * g.PGn;
    const bool thread_on = row < g.BR;

    // Item -> (c, n, band, cc), c outermost.
    auto decode = [&](int it, int &c, int &n, int &bd, int &cc) {
        cc = it % g.CC;
        int r = it / g.CC;
        bd = r % g.bands;
        r /= g.bands;
        n = r % p.N;
        c = r / p.N;
    };

    // Global chunk q of a band: band row q / cpr, chunk q % cpr starting at
    // global column cbase + 16B-chunk index.  Loads whole chunks inside the
    // row, element by element at the ragged right end, zeros outside.
    uint4 pre[kMultMaxChunks];
    auto fetch = [&](int it) {
        int c, n, bd, cc;
        decode(it, c, n, bd, cc);
        const int ih0 = bd * g.BR * p.sh - p.pbh;
        const int iw0 = cc * g.OWc * p.sw - p.pbw;
        const int cbase = (iw0 >= 0 ? iw0 / CE : -((-iw0 + CE - 1) / CE)) * CE;
        const T *plane = x + (int64_t)n * p.xs[0] + (int64_t)c * p.xs[1];
#pragma unroll
        for (int k = 0; k < kMultMaxChunks; ++k) {
            const int q = t + k * kMultThreads;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (q < g.nchunks) {
                const int br = q / g.cpr;
                const int col = cbase + (q - br * g.cpr) * CE;
                const int ih = ih0 + br;
                if (ih >= 0 && ih < p.H && col + CE > 0 && col < p.W) {
                    const T *src = plane + (int64_t)ih * p.xs[2] + col;
                    if (col >= 0 && col + CE <= p.W) {
                        v = __ldg(reinterpret_cast<const uint4 *>(src));
                    } else {
                        union { uint4 u; T e[CE]; } tmp;
#pragma unroll
                        for (int e = 0; e < CE; ++e) {
                            const int cw = col + e;
                            tmp.e[e] = (cw >= 0 && cw < p.W) ? src[e] : from_f32<T>(0.f);
                        }
                        v = tmp.u;
                    }
                }
            }
            pre[k] = v;
        }
    };

    // Widen the prefetched chunks into the shared band.  Shared column s
    // holds global column iw0 + s, so column 0 is the window start of pixel
    // group 0 and every window starts on a 16-byte boundary.  All columns a
    // stored output reads are written (zeros outside the image).
    auto deposit = [&](int it) {
        int c, n, bd, cc;
        decode(it, c, n, bd, cc);
        const int iw0 = cc * g.OWc * p.sw - p.pbw;
        const int cbase = (iw0 >= 0 ? iw0 / CE : -((-iw0 + CE - 1) / CE)) * CE;
#pragma unroll
        for (int k = 0; k < kMultMaxChunks; ++k) {
            const int q = t + k * kMultThreads;
            if (q < g.nchunks) {
                const int br = q / g.cpr;
                const int col0 = cbase + (q - br * g.cpr) * CE - iw0;   // shared column
                union { uint4 u; T e[CE]; } vals;
                vals.u = pre[k];
                float *dst = band + br * g.pitch;
#pragma unroll
                for (int e = 0; e < CE; ++e) {
                    const int sc = col0 + e;
                    if (sc >= 0 && sc < g.pitch) dst[sc] = Elem<T>::to_f32(vals.e[e]);
                }
            }
        }
    };

    fetch(i0);
    int cur_c = -1;
    for (int it = i0; it < i1; ++it) {
        int c, n, bd, cc;
        decode(it, c, n, bd, cc);
        deposit(it);
        if (c != cur_c) {
            cur_c = c;
            const int nw = g.m * p.KH * p.KW;
            for (int e = t; e < nw; e += kMultThreads) {
                const int j = e % g.m, tap = e / g.m;
                const int kh = tap / p.KW, kw = tap - kh * p.KW;
                const int co = c * g.m + j;
                wsm[e] = load_f32(w + (int64_t)co * p.ws[0] + kh * p.ws[2] + kw * p.ws[3]);
            }
            for (int j = t; j < g.m; j += kMultThreads)
                bsm[j] = p.has_bias ? load_f32(b + (int64_t)(c * g.m + j) * p.bs) : 0.f;
        }
        __syncthreads();
        if (it + 1 < i1) fetch(it + 1);   // in flight while this band is computed

        const int oh = bd * g.BR + row;
        const int ow0 = cc * g.OWc + pg * S;
        if (thread_on && oh < p.OH && ow0 < p.OW) {
            for (int mb = 0; mb < g.m; mb += MB) {
                float acc[MB][S];
#pragma unroll
                for (int j = 0; j < MB; ++j)
#pragma unroll
                    for (int i = 0; i < S; ++i) acc[j][i] = bsm[mb + j];
                for (int kh = 0; kh < p.KH; ++kh) {
                    const float4 *src = reinterpret_cast<const float4 *>(
                        band + (row * p.sh + kh) * g.pitch + pg * S * SW);
                    float xr[WIN4 * 4];
#pragma unroll
                    for (int q = 0; q < WIN4; ++q) {
                        const float4 v = src[q];
                        xr[4 * q] = v.x; xr[4 * q + 1] = v.y; xr[4 * q + 2] = v.z; xr[4 * q + 3] = v.w;
                    }
                    const float *wrow = wsm + kh * p.KW * g.m + mb;
#pragma unroll
                    for (int kw = 0; kw < kMultMaxKW; ++kw) {
                        if (kw < p.KW) {
                            float wv[MB];
                            if constexpr (MB == 4) {
                                const float4 t4 = *reinterpret_cast<const float4 *>(wrow + kw * g.m);
                                wv[0] = t4.x; wv[1] = t4.y; wv[2] = t4.z; wv[3] = t4.w;
                            } else {
#pragma unroll
                                for (int j = 0; j < MB; ++j) wv[j] = wrow[kw * g.m + j];
                            }
#pragma unroll
                            for (int j = 0; j < MB; ++j)
#pragma unroll
                                for (int i = 0; i < S; ++i)
                                    acc[j][i] = fmaf(wv[j], xr[i * SW + kw], acc[j][i]);
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < MB; ++j) {
                    T *yrow = y + (int64_t)n * p.ys[0] + (int64_t)(c * g.m + mb + j) * p.ys[1] +
                              (int64_t)oh * p.ys[2] + ow0;
                    if (g.vec_store && ow0 + S <= p.OW) {
                        union { uint4 u[S * sizeof(T) / 16]; T e[S]; } o;
#pragma unroll
                        for (int i = 0; i < S; ++i) o.e[i] = from_f32<T>(acc[j][i]);
#pragma unroll
                        for (int q = 0; q < S * (int)sizeof(T) / 16; ++q)
                            reinterpret_cast<uint4 *>(yrow)[q] = o.u[q];
                    } else {
#pragma unroll
                        for (int i = 0; i < S; ++i)
                            if (ow0 + i < p.OW) yrow[i] = from_f32<T>(acc[j][i]);
                    }
                }
            }
        }
        __syncthreads();   // the band is rewritten for the next item
    }
}

template <typename T> constexpr int mult_s() { return 16 / (int)sizeof(T); }

bool mult_geometry(const Params &p, int es, MultGeom &g) {
    g.m = p.Cout_g;
    g.S = 16 / es;
    const int CE = 16 / es;
    const int pg_need = (p.OW + g.S - 1) / g.S;
    g.CC = (pg_need + kMultThreads - 1) / kMultThreads;
    g.PGn = (pg_need + g.CC - 1) / g.CC;
    g.OWc = g.PGn * g.S;
    g.BR = kMultThreads / g.PGn;
    g.bands = (p.OH + g.BR - 1) / g.BR;
    g.rows_in = (g.BR - 1) * p.sh + p.KH;
    g.Win = (g.OWc - 1) * p.sw + p.KW;
    // every thread's window (up to 9 taps) stays inside the shared row
    const int span = (g.OWc - 1) * p.sw + kMultMaxKW;
    g.pitch = ((span > g.Win ? span : g.Win) + 3) / 4 * 4 + 4;
    g.cpr = (g.Win + CE - 1) / CE + 1;     // chunks covering the span from an aligned start
    g.nchunks = g.rows_in * g.cpr;
    if (g.nchunks > kMultThreads * kMultMaxChunks) return false;
    const int64_t items = (int64_t)p.C_in * p.N * g.bands * g.CC;
    if (items > INT32_MAX) return false;
    g.items = (int)items;
    g.ctas = g.items < 304 ? g.items : 304;   // two persistent CTAs per SM
    g.vec_store = 1;
    return true;
}

size_t mult_smem_bytes(const Params &p, const MultGeom &g) {
    return ((size_t)g.rows_in * g.pitch + (size_t)p.KH * p.KW * g.m + g.m) * sizeof(float) + 16;
}

bool mult_supports(const gconv_desc &d, const Ptrs &q) {
    if (d.Cin_g != 1 || d.Cout_g > 16) return false;
    if (d.layout != GCONV_LAYOUT_NCHW) return false;
    if (d.stride[1] != 1 && d.stride[1] != 2) return false;
    const int es = dtype_size(d.dtype);
    // 16-byte chunk loads of input rows
    if (!aligned(q.x, 16)) return false;
    if ((d.x_strides[0] * es) % 16 || (d.x_strides[1] * es) % 16 || (d.x_strides[2] * es) % 16)
        return false;
    Params p = make_params(d);
    MultGeom g;
    if (!mult_geometry(p, es, g)) return false;
    return mult_smem_bytes(p, g) <= 200 * 1024;
}

template <typename T, int SW, int MB>
cudaError_t mult_launch_t(const Params &p, const Ptrs &q, cudaStream_t s, const MultGeom &g) {
    constexpr int S = mult_s<T>();
    const size_t smem = mult_smem_bytes(p, g);
    cudaError_t e = cudaFuncSetAttribute(mult_kernel<T, SW, MB, S>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    mult_kernel<T, SW, MB, S><<<g.ctas, kMultThreads, smem, s>>>(
        static_cast<const T *>(q.x), static_cast<const T *>(q.w), static_cast<const T *>(q.b),
        static_cast<T *>(q.y), p, g);
    return cudaGetLastError();
}

template <typename T>
cudaError_t mult_launch_dtype(const Params &p, const Ptrs &q, cudaStream_t s) {
    MultGeom g;
    if (!mult_geometry(p, sizeof(T), g)) return cudaErrorNotSupported;
    // 16-byte output stores need 16-byte aligned rows
    const uintptr_t ya = reinterpret_cast<uintptr_t>(q.y);
    g.vec_store = (ya % 16 == 0) && ((p.ys[2] * (int64_t)sizeof(T)) % 16 == 0) &&
                  ((p.ys[1] * (int64_t)sizeof(T)) % 16 == 0) &&
                  ((p.ys[0] * (int64_t)sizeof(T)) % 16 == 0);
    const bool mb4 = g.m % 4 == 0;
    if (p.sw == 1)
        return mb4 ? mult_launch_t<T, 1, 4>(p, q, s, g) : mult_launch_t<T, 1, 1>(p, q, s, g);
    return mb4 ? mult_launch_t<T, 2, 4>(p, q, s, g) : mult_launch_t<T, 2, 1>(p, q, s, g);
}

cudaError_t mult_launch(const Params &p, const Ptrs &q, cudaStream_t s, int *launches) {
    *launches = 1;
    return GCONV_DISPATCH_DTYPE(p.dtype, T, [&] { return mult_launch_dtype<T>(p, q, s); });
}

}  // namespace

const Schedule kDwMult = {"dw_mult", mult_supports, mult_launch};

}  // namespace gconv
