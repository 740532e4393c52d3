// k_grp.cuh -- grp_plane: few-channel grouped convolution (1 <= Cin_g <= 8)
// with the group's weights shared by a whole CTA (executorch PR #25085,
// description, second paragraph, names this schedule: each program computes
// one output channel and the group's weights are shared).
//
// Design for sm_103a:
//  - A CTA owns one (image, group, TR x TC*P output tile); the grid runs the
//    group index fastest, so the CTAs that read the other channels of the
//    same input pixels run together and share their sectors in L2.
//  - The tile's input window ((TR-1)*SH + KH rows x (TC*P-1)*SW + KW pixels
//    x Cin_g channels) is staged raw in shared memory, CIP (4 or 8) channel
//    slots per pixel, zeros outside the image: one cp.async of Cin_g*size
//    bytes per pixel for aligned channels-last input, element loads
//    otherwise.  The group's Cout_g*Cin_g*KH*KW weights are staged as fp32
//    in [kh][kw][ci][co] order.
//  - Lanes of a warp take consecutive output rows (same column group), and
//    the staged row pitch is chosen so their 16-byte window loads fall in
//    distinct banks.  Thread (row, column group) computes P output pixels x
//    MB output channels: per kernel row it widens its (P-1)*SW + KW pixel
//    window once, then per (tap, input channel) one broadcast 16-byte weight
//    load feeds MB*P FMAs.  Kernel widths up to 9 run as a predicated,
//    fully unrolled tap loop.
//  - fp32 accumulation from the bias, one rounding per output, stores of MB
//    contiguous channels (channels-last) or per-element (NCHW).
#pragma once

#include "device_common.cuh"
#include "gconv_internal.h"
#include "launch.cuh"

namespace gconv {

constexpr int kGrpThreads = 256;
constexpr int kGrpMaxKW = 9;
// Output pixels per thread: the staged window of 4 (8) channels per pixel
// and the P x MB accumulators fit in 128 registers.
constexpr int grp_p(int cip) { return cip == 4 ? 4 : 2; }

struct GrpGeom {
    int TR, TC;           // tile rows, tile column groups (TR * TC <= 256)
    int tiles_r, tiles_c; // tiles per image along rows / columns
    int rows_in, px_in;   // staged input rows and pixels per row
    int pix_bytes;        // bytes per staged pixel = CIP * sizeof(T)
    int pitch;            // bytes per staged row
    int co_pad;           // output channels per group rounded up to MB
    int vec_load;         // one cp.async per pixel (channels-last, aligned)
    int vec_store;        // MB contiguous output channels per 16/8-byte store
    int64_t tiles;        // grid size
};

__device__ __forceinline__ void grp_cp_async(uint32_t dst, const void *src, int bytes_total,
                                             int bytes_valid) {
    // cp.async with 4, 8 or 16 bytes; zero-fill beyond bytes_valid
    if (bytes_total == 16)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                     "r"(bytes_valid));
    else if (bytes_total == 8)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;\n" ::"r"(dst), "l"(src),
                     "r"(bytes_valid));
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src),
                     "r"(bytes_valid));
}

// Widen the CIP channels of one staged pixel.
template <typename T, int CIP>
__device__ __forceinline__ void grp_widen_pixel(const unsigned char *px, float (&out)[CIP]) {
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int q = 0; q < CIP / 4; ++q) {
            const float4 v = reinterpret_cast<const float4 *>(px)[q];
            out[4 * q] = v.x; out[4 * q + 1] = v.y; out[4 * q + 2] = v.z; out[4 * q + 3] = v.w;
        }
    } else if constexpr (CIP == 4) {
        const uint2 v = *reinterpret_cast<const uint2 *>(px);
        const float2 a = unpack2(v.x, (T *)nullptr), c = unpack2(v.y, (T *)nullptr);
        out[0] = a.x; out[1] = a.y; out[2] = c.x; out[3] = c.y;
    } else {
        const uint4 v = *reinterpret_cast<const uint4 *>(px);
        const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 a = unpack2(ws[k], (T *)nullptr);
            out[2 * k] = a.x; out[2 * k + 1] = a.y;
        }
    }
}

template <typename T, int CIP, int MB, int SW>
__global__ void __launch_bounds__(kGrpThreads, 2)
grp_kernel(const T *__restrict__ x, const T *__restrict__ w, const T *__restrict__ b,
           T *__restrict__ y, Params p, GrpGeom g) {
    // Let the next kernel in the stream start launching; wait for the
    // previous kernel's memory before reading global memory.
    pdl_launch_dependents();
    pdl_wait();
    constexpr int P = grp_p(CIP);
    constexpr int PB = CIP * (int)sizeof(T);              // bytes per staged pixel
    constexpr int WPX = (P - 1) * SW + kGrpMaxKW;         // window pixels incl. unused taps
    constexpr int WBYTES = ((WPX * PB + 15) / 16) * 16;
    constexpr int WPX_LOADED = WBYTES / PB;               // pixels covered by the 16-byte loads
    extern __shared__ __align__(16) unsigned char grp_smem[];

    // Tile: group fastest, then column tile, row tile, image.
    int64_t tid = blockIdx.x;
    const int grp = (int)(tid % p.G); tid /= p.G;
    const int tcol = (int)(tid % g.tiles_c); tid /= g.tiles_c;
    const int trow = (int)(tid % g.tiles_r);
    const int n = (int)(tid / g.tiles_r);

    unsigned char *tile = grp_smem;                                      // rows_in x pitch
    float *wsm = reinterpret_cast<float *>(grp_smem + (size_t)g.rows_in * g.pitch);  // [kh][kw][ci][co_pad]
    float *bsm = wsm + p.KH * p.KW * CIP * g.co_pad;

    const int t = threadIdx.x;
    const int oh0 = trow * g.TR, ow0 = tcol * g.TC * P;
    const int ih0 = oh0 * p.sh - p.pbh, iw0 = ow0 * p.sw - p.pbw;
    const int c_first = grp * p.Cin_g;
    const T *xn = x + (int64_t)n * p.xs[0];

    // Stage the input window: pixel (r, c) -> tile + r*pitch + c*PB.
    const int npx = g.rows_in * g.px_in;
    if (g.vec_load) {
        const uint32_t base = (uint32_t)__cvta_generic_to_shared(tile);
        const int bytes = p.Cin_g * (int)sizeof(T);
        for (int e = t; e < npx; e += kGrpThreads) {
            const int r = e / g.px_in, c = e - r * g.px_in;
            const int ih = ih0 + r, iw = iw0 + c;
            const bool ok = ih >= 0 && ih < p.H && iw >= 0 && iw < p.W;
            const T *src = ok ? xn + (int64_t)ih * p.xs[2] + (int64_t)iw * p.xs[3] + c_first : x;
            grp_cp_async(base + (uint32_t)(r * g.pitch + c * PB), src, bytes, ok ? bytes : 0);
        }
        asm volatile("cp.async.commit_group;\n");
    } else {
        for (int e = t; e < npx * CIP; e += kGrpThreads) {
            const int ci = e % CIP, pe = e / CIP;
            const int r = pe / g.px_in, c = pe - r * g.px_in;
            const int ih = ih0 + r, iw = iw0 + c;
            T v = from_f32<T>(0.f);
            if (ci < p.Cin_g && ih >= 0 && ih < p.H && iw >= 0 && iw < p.W)
                v = xn[(int64_t)(c_first + ci) * p.xs[1] + (int64_t)ih * p.xs[2] +
                       (int64_t)iw * p.xs[3]];
            reinterpret_cast<T *>(tile + r * g.pitch + c * PB)[ci] = v;
        }
    }
    // Weights (zero in the padded ci / co slots) and bias.
    const int nw = p.KH * p.KW * CIP * g.co_pad;
    for (int e = t; e < nw; e += kGrpThreads) {
        const int co = e % g.co_pad;
        int r = e / g.co_pad;
        const int ci = r % CIP;
        r /= CIP;
        const int kw = r % p.KW, kh = r / p.KW;
        float v = 0.f;
        if (co < p.Cout_g && ci < p.Cin_g)
            v = load_f32(w + (int64_t)(grp * p.Cout_g + co) * p.ws[0] + (int64_t)ci * p.ws[1] +
                         (int64_t)kh * p.ws[2] + (int64_t)kw * p.ws[3]);
        wsm[e] = v;
    }
    for (int co = t; co < g.co_pad; co += kGrpThreads)
        bsm[co] = (co < p.Cout_g && p.has_bias)
                      ? load_f32(b + (int64_t)(grp * p.Cout_g + co) * p.bs) : 0.f;
    if (g.vec_load) asm volatile("cp.async.wait_group 0;\n");
    // Channel slots past Cin_g of cp.async-staged pixels are never read:
    // vector staging is used only when Cin_g == CIP.
    __syncthreads();

    const int r = t % g.TR, cg = t / g.TR;
    const int oh = oh0 + r;
    const int owt = ow0 + cg * P;
    if (cg >= g.TC || oh >= p.OH || owt >= p.OW) return;

    for (int cb = 0; cb < g.co_pad; cb += MB) {
        float acc[P][MB];
#pragma unroll
        for (int i = 0; i < P; ++i)
#pragma unroll
            for (int j = 0; j < MB; ++j) acc[i][j] = bsm[cb + j];
        for (int kh = 0; kh < p.KH; ++kh) {
            const unsigned char *src = tile + (r * p.sh + kh) * g.pitch + cg * P * SW * PB;
            float xr[WPX_LOADED][CIP];
#pragma unroll
            for (int j = 0; j < WPX_LOADED; ++j) grp_widen_pixel<T, CIP>(src + j * PB, xr[j]);
            const float *wk = wsm + (size_t)kh * p.KW * CIP * g.co_pad + cb;
#pragma unroll
            for (int kw = 0; kw < kGrpMaxKW; ++kw) {
                if (kw < p.KW) {
#pragma unroll
                    for (int ci = 0; ci < CIP; ++ci) {
                        if (ci >= p.Cin_g) break;   // padded channel slots hold zero weights
                        const float *wp = wk + (kw * CIP + ci) * g.co_pad;
                        float wv[MB];
#pragma unroll
                        for (int q = 0; q < MB / 4; ++q) {
                            const float4 t4 = reinterpret_cast<const float4 *>(wp)[q];
                            wv[4 * q] = t4.x; wv[4 * q + 1] = t4.y;
                            wv[4 * q + 2] = t4.z; wv[4 * q + 3] = t4.w;
                        }
                        if constexpr (MB < 4) {
#pragma unroll
                            for (int j = 0; j < MB; ++j) wv[j] = wp[j];
                        }
#pragma unroll
                        for (int i = 0; i < P; ++i)
#pragma unroll
                            for (int j = 0; j < MB; ++j)
                                acc[i][j] = fmaf(wv[j], xr[i * SW + kw][ci], acc[i][j]);
                    }
                }
            }
        }
        // Store: output channel grp*Cout_g + cb + j, pixel owt + i.
#pragma unroll
        for (int i = 0; i < P; ++i) {
            const int ow = owt + i;
            if (ow >= p.OW) continue;
            T *yp = y + (int64_t)n * p.ys[0] + (int64_t)oh * p.ys[2] + (int64_t)ow * p.ys[3] +
                    (int64_t)(grp * p.Cout_g + cb) * p.ys[1];
            if (g.vec_store && cb + MB <= p.Cout_g) {
                union { T e[MB]; uint32_t u[MB * sizeof(T) / 4 > 0 ? MB * sizeof(T) / 4 : 1]; } o;
#pragma unroll
                for (int j = 0; j < MB; ++j) o.e[j] = from_f32<T>(acc[i][j]);
                if constexpr (MB * sizeof(T) == 16)
                    *reinterpret_cast<uint4 *>(yp) = make_uint4(o.u[0], o.u[1], o.u[2], o.u[3]);
                else if constexpr (MB * sizeof(T) == 8)
                    *reinterpret_cast<uint2 *>(yp) = make_uint2(o.u[0], o.u[1]);
                else if constexpr (MB * sizeof(T) == 32) {
                    reinterpret_cast<uint4 *>(yp)[0] = make_uint4(o.u[0], o.u[1], o.u[2], o.u[3]);
                    reinterpret_cast<uint4 *>(yp)[1] = make_uint4(o.u[4], o.u[5], o.u[6], o.u[7]);
                } else {
#pragma unroll
                    for (int j = 0; j < MB; ++j) yp[(int64_t)j * p.ys[1]] = o.e[j];
                }
            } else {
#pragma unroll
                for (int j = 0; j < MB; ++j)
                    if (cb + j < p.Cout_g) yp[(int64_t)j * p.ys[1]] = from_f32<T>(acc[i][j]);
            }
        }
    }
}

cudaError_t grp_launch_f32(const Params &p, const Ptrs &q, cudaStream_t s);
cudaError_t grp_launch_f16(const Params &p, const Ptrs &q, cudaStream_t s);
cudaError_t grp_launch_bf16(const Params &p, const Ptrs &q, cudaStream_t s);

inline size_t grp_smem_bytes(const Params &p, const GrpGeom &g, int cip) {
    return (size_t)g.rows_in * g.pitch +
           ((size_t)p.KH * p.KW * cip * g.co_pad + g.co_pad) * sizeof(float);
}

// Launch geometry; false when the tile does not fit in shared memory.
inline bool grp_geometry(const Params &p, int es, GrpGeom &g, int &cip, int &mb) {
    cip = p.Cin_g <= 4 ? 4 : 8;
    mb = p.Cout_g <= 2 ? 2 : (p.Cout_g <= 4 ? 4 : 8);
    const int P = grp_p(cip);
    const int PB = cip * es;
    g.co_pad = (p.Cout_g + mb - 1) / mb * mb;
    g.TR = p.OH < 32 ? p.OH : 32;
    const int cg_need = (p.OW + P - 1) / P;
    g.TC = kGrpThreads / g.TR;
    if (g.TC > cg_need) g.TC = cg_need;
    g.tiles_r = (p.OH + g.TR - 1) / g.TR;
    g.tiles_c = (p.OW + g.TC * P - 1) / (g.TC * P);
    g.rows_in = (g.TR - 1) * p.sh + p.KH;
    // staged pixels: the tile's window, and every thread's 16-byte window loads
    const int sw = p.sw;
    const int wpx = (P - 1) * sw + kGrpMaxKW;
    const int wpx_loaded = ((wpx * PB + 15) / 16) * 16 / PB;
    int px = (g.TC * P - 1) * sw + p.KW;
    const int px_loads = (g.TC - 1) * P * sw + wpx_loaded;
    if (px_loads > px) px = px_loads;
    g.px_in = px;
    g.pix_bytes = PB;
    g.pitch = (px * PB + 15) / 16 * 16;
    if ((g.pitch / 16) % 2 == 0) g.pitch += 16;   // odd 16-byte slots: rows in distinct banks
    g.tiles = (int64_t)p.N * g.tiles_r * g.tiles_c * p.G;
    return grp_smem_bytes(p, g, cip) <= 200 * 1024;
}

}  // namespace gconv
