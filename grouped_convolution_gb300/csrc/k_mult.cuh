// k_mult.cuh -- dw_mult: depthwise convolution with a channel multiplier
// m <= 16 on NCHW input, every output channel of an input channel computed
// from one load of that input channel (executorch PR #25085, description,
// second paragraph, names this schedule and its multiplier bound of 16).
//
// Design for sm_103a:
//  - Work items are (input channel c, image n, band of BR output rows,
//    column chunk), column chunk fastest and c slowest, so a persistent CTA
//    restages the m*KH*KW weights only when c changes.  Items are split
//    evenly over two CTAs per SM and stepped without divisions.
//  - An item's input band ((BR-1)*SH + KH rows) arrives as one TMA tensor
//    box, two items ahead, in a two-stage ring of raw (input dtype) boxes
//    with bounded mbarrier waits; the box starts at the window's first
//    column rounded down to 16 bytes (a TMA rule) and the tensor map's zero
//    fill supplies the padding.  When x cannot be described by a tensor map
//    (unaligned base or strides) all threads fill the box with plain loads.
//  - A widening pass copies the box into a double-buffered fp32 band,
//    dropping the SHIFT columns before the first window column, so every
//    thread's window starts on a 16-byte shared boundary.  One barrier per
//    item separates the widening pass from the arithmetic.
//  - Thread (row pair, pixel group) computes S consecutive output pixels of
//    RT = 2 consecutive output rows for MB output channels at a time: each
//    band row is loaded once and multiplied into both output rows it feeds;
//    with MB = 4 the products run as packed fp32x2 FMAs over channel pairs.
//    The tap loop is unrolled for kernel widths 3, 4, 5, 7 and predicated
//    for the others.
//  - fp32 accumulation from the bias, one rounding, 16-byte stores of S
//    pixels where the row allows it.
#pragma once

#include "device_common.cuh"
#include "gconv_internal.h"
#include "launch.cuh"
#include "tma.cuh"

namespace gconv {

constexpr int kMultThreads = 256;
constexpr int kMultRT = 2;           // output rows per thread
constexpr int kMultMaxKW = 9;
constexpr int kMultCtasPerSM = 2;
constexpr int kMultSMs = 152;
constexpr int kMultSmemCap = 110 * 1024;   // two CTAs per SM
constexpr int kMultBoxMax = 256;           // TMA box extent limit

struct MultGeom {
    int m;          // multiplier (Cout_g)
    int S;          // output pixels per thread (16 bytes of T)
    int PGn;        // pixel groups per row chunk
    int TR;         // thread rows per band (each owns kMultRT output rows)
    int BR;         // output rows per band (TR * kMultRT)
    int OWc, CC;    // output columns per chunk, column chunks
    int bands;
    int rows_in;    // input rows per band
    int shift;      // first window column minus the box's first column
    int spr;        // 4-column slots per band row
    int BWX;        // box width (elements, multiple of 16 bytes)
    int pitch;      // columns per band row (multiple of 4)
    int rstride;    // fp32 elements per band row in shared memory (columns + padding)
    int stage;      // bytes per raw stage (multiple of 128)
    int band_off;   // byte offsets in shared memory
    int w_off;
    int bar_off;
    int smem;       // bytes of shared memory
    int box_bytes;  // bytes one box delivers
    int items;
    int ctas;
    int use_tma;    // x is described by a tensor map
    int vec_store;  // rows of y allow 16-byte stores of S pixels
};

// With 8 pixels per thread at column stride 1, neighbouring threads' windows
// start 32 bytes apart, so a quarter-warp's 16-byte loads hit each bank twice.
// Four padding floats after every 8 columns (column c at c + (c / 8) * 4)
// put the 8 window starts of a quarter-warp on 8 different bank quads.
constexpr bool mult_pad(int S, int SW) { return S == 8 && SW == 1; }
__host__ __device__ constexpr int mult_col(int c, bool pad) { return pad ? c + (c >> 3) * 4 : c; }

// 16-byte shared loads of a thread's window (KW = 0: any width up to 9).
template <int S, int SW, int KW>
constexpr int mult_wl4() { return ((S - 1) * SW + (KW ? KW : kMultMaxKW) + 3) / 4; }

// Band geometry for CC column chunks and at most tr_cap thread rows; false
// when the box or shared memory does not fit.
inline bool mult_band(const Params &p, int es, int CC, int tr_cap, MultGeom &g) {
    const int CE = 16 / es;                 // elements per 16 bytes
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
    if (g.rows_in > kMultBoxMax) return false;
    // Chunk cc's first window column is cc*OWc*sw - pbw; OWc*sw is a
    // multiple of CE, so its offset from the 16-byte grid does not depend on cc.
    g.shift = ((-p.pbw) % CE + CE) % CE;
    const int need = (g.OWc - 1) * p.sw + p.KW;   // band columns the outputs use
    g.spr = (need + 3) / 4;
    g.BWX = (g.shift + 4 * g.spr + CE - 1) / CE * CE;
    if (g.BWX > kMultBoxMax) return false;
    // Every thread's 16-byte window loads stay inside its band row.
    const int wl4 = ((g.S - 1) * p.sw + kMultMaxKW + 3) / 4;
    const int span = (g.PGn - 1) * g.S * p.sw + 4 * wl4;
    g.pitch = 4 * g.spr > span ? 4 * g.spr : (span + 3) / 4 * 4;
    g.rstride = mult_pad(g.S, p.sw) ? g.pitch + ((g.pitch + 7) >> 3) * 4 : g.pitch;
    g.box_bytes = g.rows_in * g.BWX * es;
    g.stage = (g.box_bytes + 127) / 128 * 128;
    g.band_off = 2 * g.stage;
    g.w_off = g.band_off + 2 * g.rows_in * g.rstride * 4;
    g.bar_off = g.w_off + ((p.KH * p.KW * g.m + g.m) * 4 + 15) / 16 * 16;
    g.smem = g.bar_off + 32;   // two mbarriers, failure flag
    return g.smem <= kMultSmemCap;
}

// Geometry for element size es: the fewest column chunks, then the most
// thread rows, that fit.  False when none does or the item count overflows.
inline bool mult_geometry(const Params &p, int es, MultGeom &g) {
    g.m = p.Cout_g;
    g.S = 16 / es;
    g.use_tma = 0;
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
    if (items > INT32_MAX - 2) return false;
    g.items = (int)items;
    const int cap = kMultSMs * kMultCtasPerSM;
    g.ctas = g.items < cap ? g.items : cap;
    return true;
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

// Round S fp32 values to T and store them at yr (S*sizeof(T) = 16 bytes):
// one 16-byte store when the row allows it, else element stores of the
// first `valid` pixels.  A failed CTA (bad) stores NaN.
template <typename T, int S, typename Get>
__device__ __forceinline__ void mult_store(T *yr, bool full, int valid, bool bad, Get raw_get) {
    auto get = [&](int i) { return bad ? __int_as_float(0x7fc00000) : raw_get(i); };
    if (full) {
        uint32_t u[4];
        if constexpr (sizeof(T) == 4) {
#pragma unroll
            for (int i = 0; i < 4; ++i) u[i] = __float_as_uint(get(i));
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) u[i] = pack2(get(2 * i), get(2 * i + 1), (T *)nullptr);
        }
        *reinterpret_cast<uint4 *>(yr) = make_uint4(u[0], u[1], u[2], u[3]);
    } else {
#pragma unroll
        for (int i = 0; i < S; ++i)
            if (i < valid) yr[i] = from_f32<T>(get(i));
    }
}

// One block of MB output channels for kMultRT output rows x S pixels of one
// thread.  brow: the thread's first window in the band (row stride pitch);
// wsm: weights [kh][kw][m] from the block's first channel; bsm: its bias;
// yr: output of the block's first channel, first row, first pixel.
// MB == 4 runs packed fp32x2 FMAs over channel pairs (the weights of two
// channels against one input value duplicated into both lanes); MB == 1
// scalar FMAs.  Both round each product-sum to nearest in fp32.
template <typename T, int SW, int MB, int KWT>
__device__ __forceinline__ void mult_block(const float *brow, int pitch, int nq, int sh, int KH,
                                           int KW, const float *wsm, int m, const float *bsm,
                                           T *yr, int64_t ys1, int64_t ys2, int rows, bool full,
                                           int valid, bool bad) {
    constexpr int S = 16 / (int)sizeof(T);
    constexpr int WL4 = mult_wl4<S, SW, KWT>();
    constexpr int KWU = KWT ? KWT : kMultMaxKW;
    constexpr int MP = MB == 4 ? 2 : 1;               // packed channel pairs
    float2 acc2[kMultRT][MP][S];                      // MB == 4
    float acc1[kMultRT][S];                           // MB == 1
    if constexpr (MB == 4) {
#pragma unroll
        for (int jp = 0; jp < MP; ++jp) {
            const float2 bj = make_float2(bsm[2 * jp], bsm[2 * jp + 1]);
#pragma unroll
            for (int rr = 0; rr < kMultRT; ++rr)
#pragma unroll
                for (int i = 0; i < S; ++i) acc2[rr][jp][i] = bj;
        }
    } else {
#pragma unroll
        for (int rr = 0; rr < kMultRT; ++rr)
#pragma unroll
            for (int i = 0; i < S; ++i) acc1[rr][i] = bsm[0];
    }
    for (int qq = 0; qq < nq; ++qq) {
        // Input row qq of this thread's rows, read once for both output rows.
        const float *src = brow + qq * pitch;
        float xr[WL4 * 4];
#pragma unroll
        for (int l = 0; l < WL4; ++l) {
            // columns 4l .. 4l+3 of the window (the window starts on a
            // multiple of 8 columns when the band is padded)
            const float4 v = *reinterpret_cast<const float4 *>(src + mult_col(4 * l, mult_pad(S, SW)));
            xr[4 * l] = v.x; xr[4 * l + 1] = v.y; xr[4 * l + 2] = v.z; xr[4 * l + 3] = v.w;
        }
#pragma unroll
        for (int rr = 0; rr < kMultRT; ++rr) {
            const int kh = qq - rr * sh;   // kernel row feeding output row rr
            if (kh < 0 || kh >= KH) continue;
            const float *wrow = wsm + kh * KW * m;
#pragma unroll
            for (int kw = 0; kw < KWU; ++kw) {
                if (!KWT && kw >= KW) break;
                if constexpr (MB == 4) {
                    const float4 t4 = *reinterpret_cast<const float4 *>(wrow + kw * m);
                    const float2 w01 = make_float2(t4.x, t4.y), w23 = make_float2(t4.z, t4.w);
#pragma unroll
                    for (int i = 0; i < S; ++i) {
                        const float xv = xr[i * SW + kw];
                        const float2 xx = make_float2(xv, xv);
                        acc2[rr][0][i] = __ffma2_rn(w01, xx, acc2[rr][0][i]);
                        acc2[rr][1][i] = __ffma2_rn(w23, xx, acc2[rr][1][i]);
                    }
                } else {
                    const float wv = wrow[kw * m];
#pragma unroll
                    for (int i = 0; i < S; ++i) acc1[rr][i] = fmaf(wv, xr[i * SW + kw], acc1[rr][i]);
                }
            }
        }
    }
#pragma unroll
    for (int rr = 0; rr < kMultRT; ++rr) {
        if (rr >= rows) break;
        T *yrow = yr + rr * ys2;
        if constexpr (MB == 4) {
#pragma unroll
            for (int jp = 0; jp < MP; ++jp) {
                mult_store<T, S>(yrow + (2 * jp) * ys1, full, valid, bad,
                                 [&](int i) { return acc2[rr][jp][i].x; });
                mult_store<T, S>(yrow + (2 * jp + 1) * ys1, full, valid, bad,
                                 [&](int i) { return acc2[rr][jp][i].y; });
            }
        } else {
            mult_store<T, S>(yrow, full, valid, bad, [&](int i) { return acc1[rr][i]; });
        }
    }
}


template <typename T, int SW, int MB, int KWT>
__global__ void __launch_bounds__(kMultThreads, kMultCtasPerSM)
mult_kernel(const __grid_constant__ CUtensorMap xmap, const T *__restrict__ x,
            const T *__restrict__ w, const T *__restrict__ b, T *__restrict__ y, Params p,
            MultGeom g) {
    // Let the next kernel in the stream start launching; wait for the
    // previous kernel's memory before reading global memory.
    pdl_launch_dependents();
    pdl_wait();
    constexpr int S = 16 / (int)sizeof(T);            // output pixels per thread
    extern __shared__ __align__(128) unsigned char mult_smem[];
    const uint32_t ring = smem_addr(mult_smem);       // raw stage s at ring + s*stage
    float *band0 = reinterpret_cast<float *>(mult_smem + g.band_off);
    float *wsm = reinterpret_cast<float *>(mult_smem + g.w_off);   // [kh][kw][m]
    float *bsm = wsm + p.KH * p.KW * g.m;                          // [m]
    const uint32_t bars = ring + (uint32_t)g.bar_off;
    volatile int *failed = reinterpret_cast<volatile int *>(mult_smem + g.bar_off + 16);
    const int KW = KWT ? KWT : p.KW;
    const int band_floats = g.rows_in * g.rstride;
    constexpr bool PAD = mult_pad(S, SW);

    const int t = threadIdx.x;
    const int per = g.items / g.ctas, extra = g.items % g.ctas;
    const int i0 = blockIdx.x * per + min((int)blockIdx.x, extra);
    const int i1 = i0 + per + ((int)blockIdx.x < extra ? 1 : 0);
    if (i0 >= i1) return;   // the same for the whole CTA

    // Box of item `it`: columns from its first window column minus shift,
    // rows from its first input row.
    auto box_x = [&](const MultItem &it) { return it.cc * g.OWc * p.sw - p.pbw - g.shift; };
    auto box_y = [&](const MultItem &it) { return it.bd * g.BR * p.sh - p.pbh; };
    int issued = 0;   // boxes issued (thread 0)
    auto issue = [&](const MultItem &it, int s) {   // one thread
        ++issued;
        const uint32_t bar = bars + 8u * s;
        mbar_arrive_expect_tx(bar, (uint32_t)g.box_bytes);
        tma_load_4d(ring + (uint32_t)(s * g.stage), &xmap, bar, box_x(it), box_y(it), it.c, it.n);
    };
    // The same box with plain loads (x without a tensor map), zeros outside.
    auto fill = [&](const MultItem &it, int s) {
        T *raw = reinterpret_cast<T *>(mult_smem + s * g.stage);
        const int x0 = box_x(it), y0 = box_y(it);
        const T *plane = x + (int64_t)it.n * p.xs[0] + (int64_t)it.c * p.xs[1];
        for (int e = t; e < g.rows_in * g.BWX; e += kMultThreads) {
            const int r = e / g.BWX, col = e - r * g.BWX;
            const int ih = y0 + r, iw = x0 + col;
            T v = from_f32<T>(0.f);
            if (ih >= 0 && ih < p.H && iw >= 0 && iw < p.W) v = plane[(int64_t)ih * p.xs[2] + iw];
            raw[e] = v;
        }
    };

    // Widening pass: band slot (r, f) = box row r, columns shift + 4f ... + 3.
    // Slots are dealt round-robin; each thread steps its slot without
    // divisions.
    const int slot_dr = kMultThreads / g.spr, slot_df = kMultThreads - slot_dr * g.spr;
    const int slot_r0 = t / g.spr, slot_f0 = t - slot_r0 * g.spr;
    auto widen_box = [&](int s, float *band) {
        const T *raw = reinterpret_cast<const T *>(mult_smem + s * g.stage) + g.shift;
        int r = slot_r0, f = slot_f0;
        while (r < g.rows_in) {
            const T *src = raw + r * g.BWX + 4 * f;
            *reinterpret_cast<float4 *>(band + r * g.rstride + mult_col(4 * f, PAD)) =
                make_float4(Elem<T>::to_f32(src[0]), Elem<T>::to_f32(src[1]),
                            Elem<T>::to_f32(src[2]), Elem<T>::to_f32(src[3]));
            f += slot_df;
            r += slot_dr;
            if (f >= g.spr) { f -= g.spr; ++r; }
        }
    };

    MultItem item;
    item.set(i0, g, p.N);
    MultItem ahead = item;   // the item two places further on
    ahead.next(g, p.N);
    if (t == 0) {
        *failed = 0;
        if (g.use_tma) {
            tma_prefetch_map(&xmap);
            mbar_init(bars, 1);
            mbar_init(bars + 8u, 1);
            fence_barrier_init();
            issue(item, 0);
            if (i0 + 1 < i1) issue(ahead, 1);
        }
    }
    ahead.next(g, p.N);
    __syncthreads();

    const int trow = t / g.PGn, pg = t - trow * g.PGn;
    const bool thread_on = trow < g.TR;
    const int brow_off = trow * kMultRT * p.sh * g.rstride + mult_col(pg * S * SW, PAD);
    const int nq = (kMultRT - 1) * p.sh + p.KH;       // band rows a thread reads

    int cur_c = -1;
    int waited = 0;   // boxes this thread has seen arrive (box k uses stage k & 1)
    bool ok = true;   // every wait of this thread so far succeeded
    for (int it = i0, k = 0; it < i1; ++it, ++k) {
        const int s = k & 1;
        float *band = band0 + s * band_floats;
        if (g.use_tma) {
            // After this thread's first failed wait nothing more is waited
            // for; the waits of the others give up once the CTA is marked
            // failed, and thread 0 issues nothing after it.
            if (ok) {
                if (mbar_wait(bars + 8u * s, (uint32_t)((k >> 1) & 1), failed)) {
                    ++waited;
                } else {
                    ok = false;
                    *failed = 1;
                }
            }
        } else {
            fill(item, s);
            __syncthreads();
        }
        widen_box(s, band);
        if (item.c != cur_c) {
            if (cur_c >= 0) __syncthreads();   // the previous item is done with wsm
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
        __syncthreads();   // band and weights ready; raw stage s is free
        // Refill stage s two items ahead (not after a failed wait).
        if (g.use_tma && t == 0 && it + 2 < i1 && !*failed) issue(ahead, s);
        ahead.next(g, p.N);
        const bool bad = *failed != 0;

        const int oh0 = item.bd * g.BR + trow * kMultRT;
        const int ow0 = item.cc * g.OWc + pg * S;
        if (thread_on && oh0 < p.OH && ow0 < p.OW) {
            T *ybase = y + (int64_t)item.n * p.ys[0] + (int64_t)(item.c * g.m) * p.ys[1] +
                       (int64_t)oh0 * p.ys[2] + ow0;
            const bool full = g.vec_store && ow0 + S <= p.OW;
            const int rows = p.OH - oh0 < kMultRT ? p.OH - oh0 : kMultRT;
            for (int mb = 0; mb < g.m; mb += MB)
                mult_block<T, SW, MB, KWT>(band + brow_off, g.rstride, nq, p.sh, p.KH, KW, wsm + mb,
                                           g.m, bsm + mb, ybase + (int64_t)mb * p.ys[1], p.ys[1],
                                           p.ys[2], rows, full, p.OW - ow0, bad);
        }
        item.next(g, p.N);
    }
    // After a failed wait, boxes issued but never seen to arrive may still be
    // landing in this CTA's shared memory: wait for each once more (bounded)
    // before the CTA exits.  Boxes k = 0 .. issued-1 went to stage k & 1.
    if (t == 0 && g.use_tma && *failed) {
        for (int q = waited; q < issued; ++q)
            (void)mbar_wait(bars + 8u * (uint32_t)(q & 1), (uint32_t)((q >> 1) & 1));
    }
}

// Host launcher for one dtype: geometry, tensor map (or plain fills),
// output-store alignment, template choice (column stride, multiplier
// blocking, kernel width).
template <typename T, int SW, int MB, int KWT>
cudaError_t mult_launch_t(const CUtensorMap &map, const Params &p, const Ptrs &q, cudaStream_t s,
                          const MultGeom &g) {
    cudaError_t e = cudaFuncSetAttribute(mult_kernel<T, SW, MB, KWT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem);
    if (e != cudaSuccess) return e;
    e = launch_kernel(mult_kernel<T, SW, MB, KWT>, dim3(g.ctas), dim3(kMultThreads), g.smem, s, map,
                   static_cast<const T *>(q.x), static_cast<const T *>(q.w),
                   static_cast<const T *>(q.b), static_cast<T *>(q.y), p, g);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename T, int MB>
cudaError_t mult_launch_kw(const CUtensorMap &map, const Params &p, const Ptrs &q, cudaStream_t s,
                           const MultGeom &g) {
    if (p.sw == 2) return mult_launch_t<T, 2, MB, 0>(map, p, q, s, g);
    switch (p.KW) {
    case 3: return mult_launch_t<T, 1, MB, 3>(map, p, q, s, g);
    case 4: return mult_launch_t<T, 1, MB, 4>(map, p, q, s, g);
    case 5: return mult_launch_t<T, 1, MB, 5>(map, p, q, s, g);
    case 7: return mult_launch_t<T, 1, MB, 7>(map, p, q, s, g);
    }
    return mult_launch_t<T, 1, MB, 0>(map, p, q, s, g);
}

template <typename T>
cudaError_t mult_launch_dtype(const Params &p, const Ptrs &q, cudaStream_t s) {
    MultGeom g;
    if (!mult_geometry(p, sizeof(T), g)) return cudaErrorNotSupported;
    const int64_t es = sizeof(T);
    CUtensorMap map{};
    const bool tma_ok = reinterpret_cast<uintptr_t>(q.x) % 16 == 0 && (p.xs[2] * es) % 16 == 0 &&
                        (p.xs[1] * es) % 16 == 0 && (p.xs[0] * es) % 16 == 0;
    if (tma_ok) {
        // x as (W, H, C, N), innermost first; a box is one item's band.
        const uint64_t dims[4] = {(uint64_t)p.W, (uint64_t)p.H, (uint64_t)p.C_in, (uint64_t)p.N};
        const uint64_t strides[3] = {(uint64_t)(p.xs[2] * es), (uint64_t)(p.xs[1] * es),
                                     (uint64_t)(p.xs[0] * es)};
        const uint32_t box[4] = {(uint32_t)g.BWX, (uint32_t)g.rows_in, 1u, 1u};
        g.use_tma = tma_encode_4d(&map, tma_dtype<T>(), q.x, dims, strides, box) ? 1 : 0;
    }
    // 16-byte output stores need 16-byte aligned rows
    const uintptr_t ya = reinterpret_cast<uintptr_t>(q.y);
    g.vec_store = (ya % 16 == 0) && ((p.ys[2] * es) % 16 == 0) && ((p.ys[1] * es) % 16 == 0) &&
                  ((p.ys[0] * es) % 16 == 0) && p.ys[3] == 1;
    return g.m % 4 == 0 ? mult_launch_kw<T, 4>(map, p, q, s, g)
                        : mult_launch_kw<T, 1>(map, p, q, s, g);
}

cudaError_t mult_launch_f32(const Params &p, const Ptrs &q, cudaStream_t s);
cudaError_t mult_launch_f16(const Params &p, const Ptrs &q, cudaStream_t s);
cudaError_t mult_launch_bf16(const Params &p, const Ptrs &q, cudaStream_t s);

}  // namespace gconv
