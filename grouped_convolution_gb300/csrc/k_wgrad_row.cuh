// k_wgrad_row.cuh -- the weight-gradient partial pass on the dw_row8 row
// ring: kernel, geometry and per-dtype launcher.  What it computes and how
// is described in k_wgrad_row.cu.
#pragma once

#include "k_row8.cuh"

namespace gconv {

struct WRowGeom {
    Row8Geom r;    // ring, chunks and thread layout (stage covers both boxes)
    int x_area;    // bytes of a stage's input box, rounded up to 128
    int gy_box;    // bytes of a stage's gy box (R rows x OWc pixels x chunk)
    int units;     // output rows per channel chunk: N * CC * OH
    int ctas;      // CTAs per channel chunk = workspace slices
};

template <typename T, int K>
bool wrow_geometry(const Params &p, WRowGeom &wg) {
    constexpr int VEC = row8_vec<T>(K);
    Row8Geom &g = wg.r;
    if (!row8_geometry<T, K>(p, g)) return false;
    const int R = (K + p.sh - 1) / p.sh;
    wg.x_area = (g.box_bytes + 127) / 128 * 128;
    wg.gy_box = g.OWc * g.pitch * R;
    g.stage = wg.x_area + (wg.gy_box + 127) / 128 * 128;
    int ns = (200 * 1024 / row8_ctas_per_sm(K) - 8 * kRow8MaxStages - 16) / g.stage;
    if (ns > kRow8MaxStages) ns = kRow8MaxStages;
    if (ns < 2) return false;
    g.NS = ns;
    // The final pixel-group sums reuse the ring.
    const int64_t red = (int64_t)(K * K + 1) * g.PG * g.CVc * VEC * 4;
    if (red > (int64_t)ns * g.stage) return false;
    const int64_t units = (int64_t)p.N * g.CC * p.OH;
    if (units > INT32_MAX / 2) return false;
    wg.units = (int)units;
    int cap = 152 * row8_ctas_per_sm(K) / g.HC;
    if (cap < 1) cap = 1;
    wg.ctas = wg.units < cap ? wg.units : cap;
    return true;
}

template <typename T, int K, int SH>
__global__ void __launch_bounds__(row8_max_threads(K), row8_ctas_per_sm(K))
wgrad_row_kernel(const __grid_constant__ CUtensorMap xmap,
                 const __grid_constant__ CUtensorMap gmap, float *__restrict__ ws, Params p,
                 WRowGeom wg) {
    pdl_launch_dependents();
    pdl_wait();
    constexpr int SW = SH;
    constexpr int VEC = row8_vec<T>(K);
    constexpr int P = VEC / 2;
    constexpr int S = row8_s(K);
    constexpr int VB = VEC * (int)sizeof(T);
    constexpr int R = (K + SH - 1) / SH;   // output rows open at once
    constexpr int U = SH * R;              // input rows per stage
    constexpr int WIN = (S - 1) * SW + K;
    constexpr int NT = K * K + 1;          // taps, then the bias
    using V = Vec<T, VEC>;
    extern __shared__ __align__(128) unsigned char wrow_ring[];
    const Row8Geom &g = wg.r;

    const int t = threadIdx.x;
    const int cvl = t % g.CVc;
    const int pg = t / g.CVc;
    const int hc = blockIdx.y;
    const int cb = g.CVc * VEC;            // channels of a chunk

    // This CTA's output rows [o0, o1) of its chunk's list.
    const int per = wg.units / (int)gridDim.x, extra = wg.units % (int)gridDim.x;
    const int o0 = (int)blockIdx.x * per + min((int)blockIdx.x, extra);
    const int o1 = o0 + per + ((int)blockIdx.x < extra ? 1 : 0);

    const uint32_t ring = smem_addr(wrow_ring);
    const uint32_t bars = ring + (uint32_t)(g.NS * g.stage);
    volatile int *abort_flag =
        reinterpret_cast<volatile int *>(wrow_ring + g.NS * g.stage + 8 * g.NS);
    const int row_bytes = g.Win * g.pitch;
    const int gy_row_bytes = g.OWc * g.pitch;
    const uint32_t tx_bytes = (uint32_t)(g.box_bytes + wg.gy_box);

    // Producer (thread 0 only).
    Row8Run prun{};
    int pnext_u = 0, pst = 0, pnst = 0, pslot = 0;
    int pissued = 0;
    bool pdone = o0 >= o1;
    auto issue = [&]() {
        if (pdone) return;
        ++pissued;
        const uint32_t bar = bars + 8u * pslot;
        const uint32_t dst = ring + (uint32_t)(pslot * g.stage);
        const int c0 = hc * cb;
        mbar_arrive_expect_tx(bar, tx_bytes);
        tma_load_4d(dst, &xmap, bar, c0, prun.cc * g.OWc * SW - p.pbw,
                    prun.oh0 * SH - p.pbh + pst * U, prun.n);
        tma_load_4d(dst + (uint32_t)wg.x_area, &gmap, bar, c0, prun.cc * g.OWc,
                    prun.oh0 + pst * R, prun.n);
        if (++pslot == g.NS) pslot = 0;
        if (++pst == pnst) {
            if (pnext_u >= o1) {
                pdone = true;
            } else {
                prun = row8_run_at<K, SH>(pnext_u, o1, p.OH, g.CC, 1);
                pnext_u += prun.rows;
                pst = 0;
                pnst = (prun.nin + U - 1) / U;
            }
        }
    };

    if (t == 0) {
        tma_prefetch_map(&xmap);
        tma_prefetch_map(&gmap);
        for (int i = 0; i < g.NS; ++i) mbar_init(bars + 8u * i, 1);
        *abort_flag = 0;
        fence_barrier_init();
        if (!pdone) {
            prun = row8_run_at<K, SH>(o0, o1, p.OH, g.CC, 1);
            pnext_u = o0 + prun.rows;
            pnst = (prun.nin + U - 1) / U;
            for (int i = 0; i < g.NS; ++i) issue();   // prologue: NS stages in flight
        }
    }
    __syncthreads();

    float2 acc[K][K][P];
    float2 accb[P];
#pragma unroll
    for (int k = 0; k < P; ++k) accb[k] = make_float2(0.f, 0.f);
#pragma unroll
    for (int a = 0; a < K; ++a)
#pragma unroll
        for (int c = 0; c < K; ++c)
#pragma unroll
            for (int k = 0; k < P; ++k) acc[a][c][k] = make_float2(0.f, 0.f);

    int cslot = 0;
    uint32_t cphase = 0;
    bool bad = false;
    int cwaited = 0;
    const uint32_t xwin0 = (uint32_t)(cvl * VB + pg * S * SW * g.pitch);
    const uint32_t gwin0 = (uint32_t)(wg.x_area + cvl * VB + pg * S * g.pitch);
    int u = o0;
    while (u < o1) {
        const Row8Run run = row8_run_at<K, SH>(u, o1, p.OH, g.CC, 1);
        u += run.rows;
        // gy set s holds the output row j of the run with j mod R == s; rows
        // before the run's first and after its last stay zero.
        float2 gyr[R][S][P];
#pragma unroll
        for (int s = 0; s < R; ++s)
#pragma unroll
            for (int i = 0; i < S; ++i)
#pragma unroll
                for (int k = 0; k < P; ++k) gyr[s][i][k] = make_float2(0.f, 0.f);

        for (int r0 = 0; r0 < run.nin; r0 += U) {
            const bool arrived = !bad && mbar_wait(bars + 8u * cslot, cphase, abort_flag);
            if (arrived) ++cwaited;
            if (t == 0 && *abort_flag) pdone = true;
            if (!arrived && !bad) {
                bad = true;
                *abort_flag = 1;
#pragma unroll
                for (int a = 0; a < K; ++a)
#pragma unroll
                    for (int c = 0; c < K; ++c)
#pragma unroll
                        for (int k = 0; k < P; ++k) acc[a][c][k] = make_float2(kNaN, kNaN);
#pragma unroll
                for (int k = 0; k < P; ++k) accb[k] = make_float2(kNaN, kNaN);
            }
            const uint32_t st = ring + (uint32_t)(cslot * g.stage);
            const int j0 = r0 / SH;   // run-relative output row of the stage's first gy row
#pragma unroll
            for (int ph = 0; ph < U; ++ph) {
                if (ph % SH == 0) {
                    // Output row j0 + ph/SH takes its first tap row here.
                    const int jr = ph / SH;
                    const bool live = j0 + jr < run.rows;
#pragma unroll
                    for (int i = 0; i < S; ++i) {
                        V v;
                        Lds<VB>::load(v, st + gwin0 + (uint32_t)(jr * gy_row_bytes + i * g.pitch));
                        widen<T, VEC>(v, gyr[jr][i]);
#pragma unroll
                        for (int k = 0; k < P; ++k) {
                            if (!live) gyr[jr][i][k] = make_float2(0.f, 0.f);
                            accb[k].x += gyr[jr][i][k].x;
                            accb[k].y += gyr[jr][i][k].y;
                        }
                    }
                }
                float2 xr[WIN][P];
#pragma unroll
                for (int j = 0; j < WIN; ++j) {
                    V v;
                    Lds<VB>::load(v, st + xwin0 + (uint32_t)(ph * row_bytes + j * g.pitch));
                    widen<T, VEC>(v, xr[j]);
                }
#pragma unroll
                for (int kh = 0; kh < K; ++kh) {
                    const int d = ph - kh;
                    if (fmod_pos(d, SH) != 0) continue;   // no output row has tap row kh here
                    const int set = fmod_pos(fdiv(d, SH), R);
#pragma unroll
                    for (int kw = 0; kw < K; ++kw)
#pragma unroll
                        for (int i = 0; i < S; ++i)
#pragma unroll
                            for (int k = 0; k < P; ++k)
                                fma2_packed(acc[kh][kw][k], gyr[set][i][k], xr[i * SW + kw][k]);
                }
            }
            if (++cslot == g.NS) {
                cslot = 0;
                cphase ^= 1u;
            }
            __syncthreads();          // every thread is done with that stage
            if (t == 0) issue();      // refill it NS stages ahead
        }
    }
    // After a failed wait, boxes issued but never seen to arrive may still be
    // landing: wait for each once more (bounded) before going on.
    if (t == 0 && *abort_flag)
        for (int q = cwaited; q < pissued; ++q)
            (void)mbar_wait(bars + 8u * (uint32_t)(q % g.NS), (uint32_t)((q / g.NS) & 1));
    __syncthreads();
    const bool failed = *abort_flag != 0;
    float *slice = ws + ((int64_t)blockIdx.x * p.C_out + (int64_t)hc * cb) * NT;
    const int nent = cb * NT;   // this chunk's entries, [channel][tap] order
    if (failed) {
        // The ring may still be written by a copy that never completed: do
        // not reuse it, report NaN for the whole chunk.
        for (int e = t; e < nent; e += blockDim.x)
            if (hc * cb + e / NT < p.C_out) slice[e] = kNaN;
        return;
    }
    // Pixel-group sums: red[tap][pg][chunk channel].
    float *red = reinterpret_cast<float *>(wrow_ring);
#pragma unroll
    for (int tp = 0; tp < NT; ++tp) {
        float *dst = red + ((int64_t)tp * g.PG + pg) * cb + cvl * VEC;
#pragma unroll
        for (int k = 0; k < P; ++k) {
            const float2 v = tp < K * K ? acc[tp / K][tp % K][k] : accb[k];
            dst[2 * k] = v.x;
            dst[2 * k + 1] = v.y;
        }
    }
    __syncthreads();
    for (int e = t; e < nent; e += blockDim.x) {
        const int cl = e / NT, tp = e - cl * NT;
        if (hc * cb + cl >= p.C_out) continue;
        float s = 0.f;
        for (int q = 0; q < g.PG; ++q) s += red[((int64_t)tp * g.PG + q) * cb + cl];
        slice[e] = s;
    }
}

template <typename T, int K, int SH>
cudaError_t wrow_launch_t(const Params &p, const void *x, const void *gy, float *ws,
                          cudaStream_t s) {
    constexpr int VEC = row8_vec<T>(K);
    WRowGeom wg;
    if (!wrow_geometry<T, K>(p, wg)) return cudaErrorNotSupported;
    const Row8Geom &g = wg.r;
    const uint64_t es = sizeof(T);
    const int R = (K + SH - 1) / SH;
    const uint64_t xd[4] = {(uint64_t)p.C_out, (uint64_t)p.W, (uint64_t)p.H, (uint64_t)p.N};
    const uint64_t xst[3] = {(uint64_t)p.xs[3] * es, (uint64_t)p.xs[2] * es, (uint64_t)p.xs[0] * es};
    const uint32_t xbox[4] = {(uint32_t)(g.CVc * VEC), (uint32_t)g.Win, (uint32_t)(SH * R), 1u};
    const uint64_t gd[4] = {(uint64_t)p.C_out, (uint64_t)p.OW, (uint64_t)p.OH, (uint64_t)p.N};
    const uint64_t gst[3] = {(uint64_t)p.ys[3] * es, (uint64_t)p.ys[2] * es, (uint64_t)p.ys[0] * es};
    const uint32_t gbox[4] = {(uint32_t)(g.CVc * VEC), (uint32_t)g.OWc, (uint32_t)R, 1u};
    CUtensorMap xmap, gmap;
    if (!tma_encode_4d(&xmap, tma_dtype<T>(), x, xd, xst, xbox)) return cudaErrorInvalidValue;
    if (!tma_encode_4d(&gmap, tma_dtype<T>(), gy, gd, gst, gbox)) return cudaErrorInvalidValue;
    const size_t smem = (size_t)g.NS * g.stage + 8 * (size_t)g.NS + 16;
    cudaError_t e = cudaFuncSetAttribute(wgrad_row_kernel<T, K, SH>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_kernel(wgrad_row_kernel<T, K, SH>, dim3(wg.ctas, g.HC), dim3(g.CVc * g.PG), smem, s,
                   xmap, gmap, ws, p, wg);
    return e != cudaSuccess ? e : cudaGetLastError();
}


// Per dtype: the slices a call writes (0: not taken) and the launch, for
// square kernels of 3, 5 or 7 at square stride 1 or 2.
template <typename T>
int wrow_slices_dtype(const Params &p) {
    WRowGeom wg;
    switch (p.KH) {
    case 3: return wrow_geometry<T, 3>(p, wg) ? wg.ctas : 0;
    case 5: return wrow_geometry<T, 5>(p, wg) ? wg.ctas : 0;
    case 7: return wrow_geometry<T, 7>(p, wg) ? wg.ctas : 0;
    }
    return 0;
}

template <typename T>
cudaError_t wrow_launch_dtype(const Params &p, const void *x, const void *gy, float *ws,
                              cudaStream_t s) {
#define GCONV_WROW_CASE(KK, SS) \
    if (p.KH == KK && p.sh == SS) return wrow_launch_t<T, KK, SS>(p, x, gy, ws, s);
    GCONV_WROW_CASE(3, 1) GCONV_WROW_CASE(3, 2)
    GCONV_WROW_CASE(5, 1) GCONV_WROW_CASE(5, 2)
    GCONV_WROW_CASE(7, 1) GCONV_WROW_CASE(7, 2)
#undef GCONV_WROW_CASE
    return cudaErrorNotSupported;
}

int wrow_slices_f32(const Params &p);
int wrow_slices_f16(const Params &p);
int wrow_slices_bf16(const Params &p);
cudaError_t wrow_launch_f32(const Params &p, const void *x, const void *gy, float *ws, cudaStream_t s);
cudaError_t wrow_launch_f16(const Params &p, const void *x, const void *gy, float *ws, cudaStream_t s);
cudaError_t wrow_launch_bf16(const Params &p, const void *x, const void *gy, float *ws, cudaStream_t s);

}  // namespace gconv
