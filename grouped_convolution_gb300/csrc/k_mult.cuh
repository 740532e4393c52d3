// k_mult.cuh -- dw_mult: depthwise convolution with a channel multiplier
// m <= 16 on NCHW input, every output channel of an input channel computed
// from one load of that input channel (executorch PR #25085, description,
// second paragraph: all output channels of an input channel per load, for
// multipliers up to 16).
//
// Design for sm_103a:
//  - Work items are (input channel c, image n, band of BR output rows,
//    column chunk), column chunk fastest and c slowest, so a persistent CTA
//    restages the m*KH*KW weights only when c changes.  Items are split
//    evenly over two CTAs per SM and stepped without divisions.
//  - The band's input rows ((BR-1)*SH + KH rows) are fetched one item ahead
//    as 16-byte chunks aligned in global memory (zeros outside the image)
//    into registers, then widened once to fp32 into shared memory with
//    16-byte stores.  Shared column 0 is the first window column rounded
//    down to a multiple of 4, so chunks land on 16-byte shared boundaries;
//    every thread's window then starts MIS (0..3, the same for every thread
//    and item) columns past a 16-byte boundary, and MIS is a template
//    parameter of the tap loop, so the window is read with 16-byte loads and
//    the taps index registers at compile-time offsets.
//  - Thread (row pair, pixel group) computes S consecutive output pixels of
//    RT = 2 consecutive output rows for MB output channels at a time: each
//    staged input row is loaded once and multiplied into both output rows
//    it feeds; per tap one broadcast shared load of MB weights feeds MB*S
//    FMAs per output row.
//  - fp32 accumulation from the bias, one rounding, 16-byte stores of S
//    pixels where the row allows it.
#pragma once

#include "device_common.cuh"
#include "gconv_internal.h"

namespace gconv {

constexpr int kMultThreads = 256;
constexpr int kMultRT = 2;           // output rows per thread
constexpr int kMultMaxChunks = 4;    // 16-byte global chunks per thread per band
constexpr int kMultMaxKW = 9;
constexpr int kMultCtasPerSM = 2;
constexpr int kMultSMs = 152;

struct MultGeom {
    int m;          // multiplier (Cout_g)
    int S;          // output pixels per thread (16 bytes of T)
    int PGn;        // pixel groups per row chunk
    int TR;         // thread rows per band (each owns kMultRT output rows)
    int BR;         // output rows per band (TR * kMultRT)
    int OWc, CC;    // output columns per chunk, column chunks
    int bands;
    int rows_in;    // input rows per band
    int mis;        // first window column minus shared column 0 (0..3)
    int coff;       // shared column 0 minus the first chunk's column (0 or 4)
    int cpr;        // 16-byte global chunks per band row
    int nchunks;    // chunks per band
    int pitch;      // fp32 elements per shared row (multiple of 4)
    int items;
    int ctas;
    int vec_load;   // rows of x allow 16-byte chunk loads
    int vec_store;  // rows of y allow 16-byte stores of S pixels
};

// 16-byte shared loads a thread's window needs at most.
template <int S, int SW, int MIS>
constexpr int mult_wl4() { return (MIS + (S - 1) * SW + kMultMaxKW + 3) / 4; }

inline int mult_floor_div(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

// Geometry for element size es; false when the band does not fit the
// per-thread chunk budget or the item count overflows.
// Band geometry for CC column chunks and at most tr_cap thread rows; false
// when the band's chunks exceed the per-thread budget.
inline bool mult_band(const Params &p, int es, int CC, int tr_cap, MultGeom &g) {
    const int CE = 16 / es;                 // elements per 16-byte chunk
    const int pg_need = (p.OW + g.S - 1) / g.S;
    g.CC = CC;
    g.PGn = (pg_need + CC - 1) / CC;
    g.OWc = g.PGn * g.S;
    int tr_max = kMultThreads / g.PGn;
    if (tr_max > tr_cap) tr_max = tr_cap;
    if (tr_max < 1) return false;
    const int rows_max = tr_max * kMultRT;
    // Even bands: as many as the thread rows need, each as short as possible.
    g.bands = (p.OH + rows_max - 1) / rows_max;
    const int br = (p.OH + g.bands - 1) / g.bands;
    g.TR = (br + kMultRT - 1) / kMultRT;
    g.BR = g.TR * kMultRT;
    g.bands = (p.OH + g.BR - 1) / g.BR;
    g.rows_in = (g.BR - 1) * p.sh + p.KH;
    // Window of column chunk cc starts at iw0 = cc*OWc*sw - pbw; OWc*sw is a
    // multiple of CE (and of 4), so mis and coff do not depend on cc.
    const int iw0 = -p.pbw;
    const int origin = mult_floor_div(iw0, 4) * 4;
    g.mis = iw0 - origin;
    const int cbase = mult_floor_div(origin, CE) * CE;
    g.coff = origin - cbase;
    const int need = g.mis + (g.OWc - 1) * p.sw + p.KW;   // shared columns used
    g.cpr = (g.coff + need + CE - 1) / CE;
    g.nchunks = g.rows_in * g.cpr;
    if (g.nchunks > kMultThreads * kMultMaxChunks) return false;
    // Every thread's 16-byte window loads stay inside the row.
    const int wl4 = (3 + (g.S - 1) * p.sw + kMultMaxKW + 3) / 4;
    const int span = (g.PGn - 1) * g.S * p.sw + 4 * wl4;
    g.pitch = ((need > span ? need : span) + 3) / 4 * 4;
    return true;
}

// Geometry for element size es: the fewest column chunks, then the most
// thread rows, whose band fits the chunk budget.  False when none does or
// the item count overflows.
inline bool mult_geometry(const Params &p, int es, MultGeom &g) {
    g.m = p.Cout_g;
    g.S = 16 / es;
    g.vec_load = 0;
    g.vec_store = 0;
    const int pg_need = (p.OW + g.S - 1) / g.S;
    bool ok = false;
    for (int CC = (pg_need + kMultThreads - 1) / kMultThreads; CC <= pg_need && !ok; ++CC) {
        for (int tr = kMultThreads; tr >= 1 && !ok; tr = tr > 1 ? tr / 2 : 0)
            ok = mult_band(p, es, CC, tr, g);
        if (!ok && CC >= 64) break;
    }
    if (!ok) return false;
    const int64_t items = (int64_t)p.C_in * p.N * g.bands * g.CC;
    if (items > INT32_MAX) return false;
    g.items = (int)items;
    const int cap = kMultSMs * kMultCtasPerSM;
    g.ctas = g.items < cap ? g.items : cap;
    return true;
}

inline size_t mult_smem_bytes(const Params &p, const MultGeom &g) {
    return ((size_t)g.rows_in * g.pitch + (size_t)p.KH * p.KW * g.m + g.m) * sizeof(float);
}

// Division-free cursor over items (cc fastest, then band, image, channel).
struct MultItem {
    int c, n, bd, cc;
    __device__ __forceinline__ void set(int it, const MultGeom &g, int N) {
        cc = it % g.CC;
        int r = it / g.CC;
        bd = r % g.bands;
        r /= g.bands;
        n = r % N;
        c = r / N;
    }
    __device__ __forceinline__ void next(const MultGeom &g, int N) {
        if (++cc < g.CC) return;
        cc = 0;
        if (++bd < g.bands) return;
        bd = 0;
        if (++n < N) return;
        n = 0;
        ++c;
    }
};

// Widen a 16-byte chunk of T into CE fp32 values.
template <typename T>
__device__ __forceinline__ void mult_widen(const uint4 &v, float (&f)[16 / sizeof(T)]) {
    if constexpr (sizeof(T) == 4) {
        f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
    } else {
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 a = unpack2(u[k], (T *)nullptr);
            f[2 * k] = a.x; f[2 * k + 1] = a.y;
        }
    }
}

}  // namespace gconv

namespace gconv {

template <typename T, int SW, int MB, int MIS>
__global__ void __launch_bounds__(kMultThreads, kMultCtasPerSM)
mult_kernel(const T *__restrict__ x, const T *__restrict__ w, const T *__restrict__ b,
            T *__restrict__ y, Params p, MultGeom g) {
    constexpr int CE = 16 / (int)sizeof(T);           // elements per 16-byte chunk
    constexpr int S = CE;                             // output pixels per thread
    constexpr int WL4 = mult_wl4<S, SW, MIS>();       // 16-byte window loads
    extern __shared__ __align__(16) float mult_smem[];
    float *band = mult_smem;                          // rows_in x pitch
    float *wsm = band + g.rows_in * g.pitch;          // [kh][kw][m]
    float *bsm = wsm + p.KH * p.KW * g.m;             // [m]

    const int t = threadIdx.x;
    const int per = g.items / g.ctas, extra = g.items % g.ctas;
    const int i0 = blockIdx.x * per + min((int)blockIdx.x, extra);
    const int i1 = i0 + per + ((int)blockIdx.x < extra ? 1 : 0);
    if (i0 >= i1) return;   // the same for the whole CTA

    // This thread's chunks of a band, fixed for every item: band row in the
    // high half, chunk index in the low half; -1 when the chunk is unused.
    int chunk[kMultMaxChunks];
#pragma unroll
    for (int k = 0; k < kMultMaxChunks; ++k) {
        const int q = t + k * kMultThreads;
        const int br = q / g.cpr;
        chunk[k] = q < g.nchunks ? (br << 16) | (q - br * g.cpr) : -1;
    }

    uint4 pre[kMultMaxChunks];
    // Load the band of `it` into registers: whole 16-byte chunks inside the
    // row (when rows are 16-byte aligned), element by element at a ragged
    // edge or on unaligned rows, zeros outside the image.
    auto fetch = [&](const MultItem &it) {
        const int ih0 = it.bd * g.BR * p.sh - p.pbh;
        const int cbase = it.cc * g.OWc * p.sw - p.pbw - g.mis - g.coff;
        const T *plane = x + (int64_t)it.n * p.xs[0] + (int64_t)it.c * p.xs[1];
#pragma unroll
        for (int k = 0; k < kMultMaxChunks; ++k) {
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            const int ih = ih0 + (chunk[k] >> 16);
            const int col = cbase + (chunk[k] & 0xffff) * CE;
            if (chunk[k] >= 0 && ih >= 0 && ih < p.H && col + CE > 0 && col < p.W) {
                const T *row = plane + (int64_t)ih * p.xs[2];
                if (g.vec_load && col >= 0 && col + CE <= p.W) {
                    v = __ldg(reinterpret_cast<const uint4 *>(row + col));
                } else {
                    union { uint4 u; T e[CE]; } tmp;
#pragma unroll
                    for (int e = 0; e < CE; ++e) {
                        const int cw = col + e;
                        tmp.e[e] = (cw >= 0 && cw < p.W) ? row[cw] : from_f32<T>(0.f);
                    }
                    v = tmp.u;
                }
            }
            pre[k] = v;
        }
    };
    // Widen the fetched chunks into the band: 16-byte shared stores at the
    // same place for every item (chunk index * CE - coff).
    auto deposit = [&]() {
#pragma unroll
        for (int k = 0; k < kMultMaxChunks; ++k) {
            if (chunk[k] >= 0) {
                float f[CE];
                mult_widen<T>(pre[k], f);
                const int sc0 = (chunk[k] & 0xffff) * CE - g.coff;
                float *dst = band + (chunk[k] >> 16) * g.pitch;
#pragma unroll
                for (int h = 0; h < CE / 4; ++h) {
                    const int sc = sc0 + 4 * h;
                    if (sc >= 0 && sc + 4 <= g.pitch)
                        *reinterpret_cast<float4 *>(dst + sc) =
                            make_float4(f[4 * h], f[4 * h + 1], f[4 * h + 2], f[4 * h + 3]);
                }
            }
        }
    };

    const int trow = t / g.PGn, pg = t - trow * g.PGn;
    const bool thread_on = trow < g.TR;
    const float *brow0 = band + trow * kMultRT * p.sh * g.pitch + pg * S * SW;
    const int nq = (kMultRT - 1) * p.sh + p.KH;       // input rows a thread reads

    MultItem item;
    item.set(i0, g, p.N);
    fetch(item);
    int cur_c = -1;
    for (int it = i0; it < i1; ++it) {
        deposit();
        if (item.c != cur_c) {
            cur_c = item.c;
            const int nw = g.m * p.KH * p.KW;
            for (int e = t; e < nw; e += kMultThreads) {
                const int j = e % g.m, tap = e / g.m;
                const int kh = tap / p.KW, kw = tap - kh * p.KW;
                wsm[e] = load_f32(w + (int64_t)(cur_c * g.m + j) * p.ws[0] +
                                  (int64_t)kh * p.ws[2] + (int64_t)kw * p.ws[3]);
            }
            for (int j = t; j < g.m; j += kMultThreads)
                bsm[j] = p.has_bias ? load_f32(b + (int64_t)(cur_c * g.m + j) * p.bs) : 0.f;
        }
        __syncthreads();
        MultItem nxt = item;
        nxt.next(g, p.N);
        if (it + 1 < i1) fetch(nxt);   // in flight while this band is computed

        const int oh0 = item.bd * g.BR + trow * kMultRT;
        const int ow0 = item.cc * g.OWc + pg * S;
        if (thread_on && oh0 < p.OH && ow0 < p.OW) {
            for (int mb = 0; mb < g.m; mb += MB) {
                float acc[kMultRT][MB][S];
#pragma unroll
                for (int j = 0; j < MB; ++j) {
                    const float bj = bsm[mb + j];
#pragma unroll
                    for (int rr = 0; rr < kMultRT; ++rr)
#pragma unroll
                        for (int i = 0; i < S; ++i) acc[rr][j][i] = bj;
                }
                for (int qq = 0; qq < nq; ++qq) {
                    // Input row qq of this thread's rows, read once.
                    const float4 *src = reinterpret_cast<const float4 *>(brow0 + qq * g.pitch);
                    float xr[WL4 * 4];
#pragma unroll
                    for (int l = 0; l < WL4; ++l) {
                        const float4 v = src[l];
                        xr[4 * l] = v.x; xr[4 * l + 1] = v.y; xr[4 * l + 2] = v.z; xr[4 * l + 3] = v.w;
                    }
#pragma unroll
                    for (int rr = 0; rr < kMultRT; ++rr) {
                        const int kh = qq - rr * p.sh;   // kernel row feeding output row rr
                        if (kh >= 0 && kh < p.KH) {
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
                                            acc[rr][j][i] =
                                                fmaf(wv[j], xr[MIS + i * SW + kw], acc[rr][j][i]);
                                }
                            }
                        }
                    }
                }
#pragma unroll
                for (int rr = 0; rr < kMultRT; ++rr) {
                    const int oh = oh0 + rr;
                    if (oh >= p.OH) continue;
#pragma unroll
                    for (int j = 0; j < MB; ++j) {
                        T *yrow = y + (int64_t)item.n * p.ys[0] +
                                  (int64_t)(item.c * g.m + mb + j) * p.ys[1] +
                                  (int64_t)oh * p.ys[2] + ow0;
                        if (g.vec_store && ow0 + S <= p.OW) {
                            union { uint4 u; T e[S]; } o;
#pragma unroll
                            for (int i = 0; i < S; ++i) o.e[i] = from_f32<T>(acc[rr][j][i]);
                            *reinterpret_cast<uint4 *>(yrow) = o.u;
                        } else {
#pragma unroll
                            for (int i = 0; i < S; ++i)
                                if (ow0 + i < p.OW) yrow[i] = from_f32<T>(acc[rr][j][i]);
                        }
                    }
                }
            }
        }
        __syncthreads();   // the band and weights are rewritten for the next item
        item = nxt;
    }
}

// Host launcher for one dtype: geometry, output-store alignment, template
// choice (column stride, multiplier blocking, window offset).
template <typename T, int SW, int MB, int MIS>
cudaError_t mult_launch_t(const Params &p, const Ptrs &q, cudaStream_t s, const MultGeom &g) {
    const size_t smem = mult_smem_bytes(p, g);
    cudaError_t e = cudaFuncSetAttribute(mult_kernel<T, SW, MB, MIS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    mult_kernel<T, SW, MB, MIS><<<g.ctas, kMultThreads, smem, s>>>(
        static_cast<const T *>(q.x), static_cast<const T *>(q.w), static_cast<const T *>(q.b),
        static_cast<T *>(q.y), p, g);
    return cudaGetLastError();
}

template <typename T, int SW, int MB>
cudaError_t mult_launch_mis(const Params &p, const Ptrs &q, cudaStream_t s, const MultGeom &g) {
    switch (g.mis) {
    case 0: return mult_launch_t<T, SW, MB, 0>(p, q, s, g);
    case 1: return mult_launch_t<T, SW, MB, 1>(p, q, s, g);
    case 2: return mult_launch_t<T, SW, MB, 2>(p, q, s, g);
    case 3: return mult_launch_t<T, SW, MB, 3>(p, q, s, g);
    }
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t mult_launch_dtype(const Params &p, const Ptrs &q, cudaStream_t s) {
    MultGeom g;
    if (!mult_geometry(p, sizeof(T), g)) return cudaErrorNotSupported;
    const uintptr_t xa = reinterpret_cast<uintptr_t>(q.x);
    g.vec_load = (xa % 16 == 0) && ((p.xs[2] * (int64_t)sizeof(T)) % 16 == 0) &&
                 ((p.xs[1] * (int64_t)sizeof(T)) % 16 == 0) &&
                 ((p.xs[0] * (int64_t)sizeof(T)) % 16 == 0);
    // 16-byte output stores need 16-byte aligned rows
    const uintptr_t ya = reinterpret_cast<uintptr_t>(q.y);
    g.vec_store = (ya % 16 == 0) && ((p.ys[2] * (int64_t)sizeof(T)) % 16 == 0) &&
                  ((p.ys[1] * (int64_t)sizeof(T)) % 16 == 0) &&
                  ((p.ys[0] * (int64_t)sizeof(T)) % 16 == 0) && p.ys[3] == 1;
    const bool mb4 = g.m % 4 == 0;
    if (p.sw == 1)
        return mb4 ? mult_launch_mis<T, 1, 4>(p, q, s, g) : mult_launch_mis<T, 1, 1>(p, q, s, g);
    return mb4 ? mult_launch_mis<T, 2, 4>(p, q, s, g) : mult_launch_mis<T, 2, 1>(p, q, s, g);
}

cudaError_t mult_launch_f32(const Params &p, const Ptrs &q, cudaStream_t s);
cudaError_t mult_launch_f16(const Params &p, const Ptrs &q, cudaStream_t s);
cudaError_t mult_launch_bf16(const Params &p, const Ptrs &q, cudaStream_t s);

}  // namespace gconv
