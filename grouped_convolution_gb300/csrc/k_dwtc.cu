// k_dwtc.cu -- dw_tc: depthwise convolution of NCHW bf16/fp16 planes at
// stride 1 on the tcgen05 tensor cores, the kernel's columns as a banded
// matrix.
//
// The operation is the depthwise case of the direct stencil of executorch
// PR #25085 (description, second paragraph): y[n, c*m + j, oh, ow] =
// sum_{kh, kw} w[c*m + j, 0, kh, kw] * x[n, c, oh - pad_h + kh, ow - pad_w + kw].
// This form of it is written for sm_103a.  For one input channel c, one
// kernel row kh and a tile of 16 output columns starting at ow0:
//   D[r][mm*16 + jj] += sum_k A[r][k] * B[mm*16 + jj][k]
// with A[r][k] = x[c, oh0 + r - pad_h + kh, kstart + k] (a row of the input
// plane: M = 128 output rows, K = the input columns kstart .. kstart + 31,
// kstart = ow0 - pad_w - a rounded down to a multiple of 8) and the banded
// B[mm*16 + jj][k] = w[c*m + mm, 0, kh, k - a - jj] (zero outside the
// kernel).  The m output channels of the input channel share A (N = 16 m).
// Summed over kh (tensor-memory accumulation), D[r][mm*16 + jj] is the
// output at row oh0 + r, column ow0 + jj, channel c*m + mm: the drain only
// adds the bias and rounds, no sums across rows.
//  - Staging: a unit is one channel plane of one image, 128 output rows
//    and up to 128 output columns.  Its input is loaded by TMA as 8-column
//    chunks, chunk i holding input columns base + 8i .. base + 8i + 7 of
//    the unit's R = 128 + KH - 1 rows, row after row (16 bytes a row), in
//    its own 128-byte-aligned slot: the K-major, unswizzled operand layout,
//    each chunk one K half.  The tensor
//    map's zero fill gives the padding.
//  - The 16-column tile t reads chunks 2t + 2s, 2t + 2s + 1 for K step s
//    (the leading byte offset is one chunk) from row kh on.
//  - Weights: per input channel, KH x ksteps banded matrices of N x 16,
//    built by the drain warps when the channel changes.
//  - One CTA per SM: eight warps stage the weights and drain tensor memory
//    (two warpgroups taking alternate tiles), two warps issue the MMAs of
//    alternate tiles, one warp issues the input boxes.  Two unit buffers
//    and up to eight tensor-memory tile buffers; three unit buffers.
//  - Every mbarrier wait is bounded; a wait that gives up marks the CTA
//    failed, its outputs are written as NaN, and before exiting the CTA
//    waits (bounded) for its copies and MMAs in flight before it frees its
//    tensor memory.
#include <cstdint>

#include "device_common.cuh"
#include "gconv_internal.h"
#include "launch.cuh"
#include "tc_common.cuh"
#include "tma.cuh"

namespace gconv {
namespace {

using namespace tc;

constexpr int kDWarps = 8;                    // weight staging + drain
constexpr int kDDrain = 32 * kDWarps;
constexpr int kDIssuers = 2;                  // MMA issue warps
constexpr int kDLoader = kDWarps + kDIssuers;   // the warp that issues the input boxes
constexpr int kDThreads = kDDrain + 32 * (kDIssuers + 1);
constexpr int kDMaxBufs = 8;                  // tensor-memory tile buffers
constexpr int kDUnitBufs = 3;                 // unit buffers (input staging ring)
constexpr int kDMaxTiles = 8;                 // 16-column tiles per unit
constexpr int kDSmemCap = 220 * 1024;

struct DtcGeom {
    int m, N;          // multiplier, MMA N = 16 m
    int a;             // (-pad_w) mod 8: the band's offset in its K window
    int ksteps;        // K = 16 steps per kernel row
    int owt;           // 16-column tiles per unit
    int gws, ots;      // column groups, 128-row tiles
    int R;             // staged rows per unit
    int nch;           // staged 8-column chunks per unit
    int chunk_bytes;   // one chunk's slot: R rows of 16 bytes, rounded up to 128
    int unit_bytes, b_bytes;
    int units, ctas, bufs, tmem_cols;
    int b_off0, bar_off, smem;   // weight buffers at b_off0 + i * b_bytes
    uint32_t idesc;
    int vec_store;     // 32-byte stores of 16 output columns
};

bool dwtc_geometry(const Params &p, DtcGeom &g) {
    if (p.transposed || p.sh != 1 || p.sw != 1 || p.dh != 1 || p.dw != 1) return false;
    if (p.Cin_g != 1) return false;
    if (p.dtype != GCONV_BF16 && p.dtype != GCONV_F16) return false;
    if (p.KH < 1 || p.KH > 9 || p.KW < 1 || p.KW > 9) return false;
    g.m = p.Cout_g;
    if (g.m != 1 && g.m != 2 && g.m != 4 && g.m != 8 && g.m != 16) return false;
    g.N = 16 * g.m;
    g.a = ((-p.pbw) % 8 + 8) % 8;
    g.ksteps = (g.a + 15 + p.KW - 1) / 16 + 1;   // 1 or 2 (KW <= 9)
    const int tiles = (p.OW + 15) / 16;
    g.gws = (tiles + kDMaxTiles - 1) / kDMaxTiles;
    g.owt = (tiles + g.gws - 1) / g.gws;
    g.ots = (p.OH + 127) / 128;
    g.R = 128 + p.KH - 1;
    g.nch = 2 * (g.owt - 1) + 2 * g.ksteps;
    g.chunk_bytes = (g.R * 16 + 127) / 128 * 128;   // TMA destinations 128-byte aligned
    g.unit_bytes = (g.nch * g.chunk_bytes + 127) / 128 * 128;
    g.b_bytes = (p.KH * g.ksteps * g.N * 32 + 127) / 128 * 128;
    g.b_off0 = kDUnitBufs * g.unit_bytes;   // unit buffer i at i * unit_bytes
    g.bar_off = g.b_off0 + 2 * g.b_bytes;
    g.bufs = 512 / g.N < kDMaxBufs ? 512 / g.N : kDMaxBufs;
    g.smem = g.bar_off + 8 * (2 * kDUnitBufs + 2 * kDMaxBufs + 2) + 16;
    if (g.smem > kDSmemCap) return false;
    int cols = g.bufs * g.N, pow2 = 32;
    while (pow2 < cols) pow2 *= 2;
    g.tmem_cols = pow2;
    const int64_t units = (int64_t)p.C_in * p.N * g.ots * g.gws;
    if (units > INT32_MAX) return false;
    g.units = (int)units;
    g.ctas = g.units < 152 ? g.units : 152;
    g.idesc = s_idesc(p.dtype == GCONV_BF16, 128, g.N);
    g.vec_store = 0;
    return true;
}

// Division-free cursor over units (column group fastest, then image, row
// tile, channel): consecutive units of a CTA share the channel's weights.
struct DtcUnit {
    int gw, n, ot, c;
    __device__ __forceinline__ void set(int u, const DtcGeom &g, int N) {
        gw = u % g.gws;
        int r = u / g.gws;
        n = r % N;
        r /= N;
        ot = r % g.ots;
        c = r / g.ots;
    }
    __device__ __forceinline__ void next(const DtcGeom &g, int N) {
        if (++gw < g.gws) return;
        gw = 0;
        if (++n < N) return;
        n = 0;
        if (++ot < g.ots) return;
        ot = 0;
        ++c;
    }
};

// T: element type.
template <typename T>
__global__ void __launch_bounds__(kDThreads, 1)
dwtc_kernel(const __grid_constant__ CUtensorMap xmap, const T *__restrict__ w,
            const T *__restrict__ b, T *__restrict__ y, Params p, DtcGeom g) {
    pdl_launch_dependents();
    pdl_wait();
    extern __shared__ __align__(1024) unsigned char d_smem[];
    const uint32_t sbase = smem_addr(d_smem);
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int per = g.units / g.ctas, extra = g.units % g.ctas;
    const int u0 = blockIdx.x * per + min((int)blockIdx.x, extra);
    const int nunits = per + ((int)blockIdx.x < extra ? 1 : 0);
    if (nunits <= 0) return;

    // mbarriers: staged[3] (a unit's boxes landed), free[3] (every MMA that
    // read the unit buffer completed: one commit per issuer), full[bufs] (a
    // tile's MMAs completed), empty[bufs] (a tile drained: 128 arrivals),
    // b_ready[2] (a channel's weights written into weight buffer i).  Unit
    // k uses unit buffer k % 3, in phase (k / 3) & 1.
    const uint32_t bar_staged = sbase + (uint32_t)g.bar_off;
    const uint32_t bar_free = bar_staged + 8u * kDUnitBufs;
    const uint32_t bar_full = bar_free + 8u * kDUnitBufs;
    const uint32_t bar_empty = bar_full + 8u * kDMaxBufs;
    const uint32_t bar_bready = bar_empty + 8u * kDMaxBufs;
    const int slot_off = g.bar_off + 8 * (2 * kDUnitBufs + 2 * kDMaxBufs + 2);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(d_smem + slot_off);
    volatile int *failed = reinterpret_cast<volatile int *>(d_smem + slot_off + 4);

    if (warp == kDWarps) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                         sbase + (uint32_t)slot_off),
                     "r"(g.tmem_cols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
    }
    if (t == 0) {
        for (int i = 0; i < kDUnitBufs; ++i) {
            mbar_init(bar_staged + 8u * i, 1);
            mbar_init(bar_free + 8u * i, kDIssuers);
        }
        for (int i = 0; i < 2; ++i) mbar_init(bar_bready + 8u * i, kDDrain);
        for (int i = 0; i < kDMaxBufs; ++i) {
            mbar_init(bar_full + 8u * i, 1);
            mbar_init(bar_empty + 8u * i, kDDrain / 2);
        }
        *failed = 0;
        fence_barrier_init();
        tma_prefetch_map(&xmap);
    }
    s_fence_before();
    __syncthreads();
    s_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == kDLoader) {
        // ------ input boxes: unit k into unit buffer k % 3 once the tensor
        // core has read the unit three back; the whole warp runs the loop,
        // lane 0 issues ------
        const uint32_t unit_tx = (uint32_t)(g.nch * g.R * 16);   // the boxes' bytes
        DtcUnit u;
        u.set(u0, g, p.N);
        for (int k = 0; k < nunits; ++k, u.next(g, p.N)) {
            const int ub = k % kDUnitBufs;
            if (k >= kDUnitBufs)
                s_wait_warp(bar_free + 8u * ub, (uint32_t)((k / kDUnitBufs - 1) & 1), failed);
            s_expect_tx_lane0(bar_staged + 8u * ub, unit_tx, (uint32_t)lane);
            const int col0 = 16 * g.owt * u.gw - p.pbw - g.a;   // a multiple of 8
            const int row0 = 128 * u.ot - p.pbh;
            const uint32_t ring = sbase + (uint32_t)(ub * g.unit_bytes);
            for (int i = 0; i < g.nch; ++i)
                s_tma_lane0(ring + (uint32_t)(i * g.chunk_bytes), &xmap, bar_staged + 8u * ub,
                            col0 + 8 * i, row0, u.c, u.n, (uint32_t)lane);
        }
    } else if (warp >= kDWarps) {
        // ------ MMA issue: issuer i takes tiles i, i + 2, ... ------
        const int iss = warp - kDWarps;
        int gt = 0;
        DtcUnit u;
        u.set(u0, g, p.N);
        int prev_c = -1, bsel = 1, bstaged = 0;   // bit i: phase of b_ready[i]
        for (int k = 0; k < nunits; ++k, u.next(g, p.N)) {
            const int ub = k % kDUnitBufs;
            if (u.c != prev_c) {   // the weights of a new channel, in the other buffer
                prev_c = u.c;
                bsel ^= 1;
                s_wait_warp(bar_bready + 8u * bsel, (uint32_t)((bstaged >> bsel) & 1), failed);
                bstaged ^= 1 << bsel;
            }
            s_wait_warp(bar_staged + 8u * ub, (uint32_t)((k / kDUnitBufs) & 1), failed);
            s_fence_after();
            const uint64_t ad0 = s_desc(sbase + (uint32_t)(ub * g.unit_bytes), (uint32_t)g.chunk_bytes, 128);
            const uint64_t bd0 = s_desc(sbase + (uint32_t)(g.b_off0 + bsel * g.b_bytes), 128, 256);
            for (int tt = 0; tt < g.owt; ++tt, ++gt) {
                if (gt % kDIssuers != iss) continue;
                const int tb = gt % g.bufs;
                const int use = gt / g.bufs;
                if (use >= 1) s_wait_warp(bar_empty + 8u * tb, (uint32_t)((use - 1) & 1), failed);
                s_fence_after();
                if (!__any_sync(0xffffffffu, *failed != 0)) {
                    const uint32_t d = tmem + (uint32_t)(tb * g.N);
                    // A: chunks 2tt + 2s (K 0-7) and the next (K 8-15) from
                    // staged row kh on; the descriptors' start fields (16-byte
                    // units, no carry below 2^18 bytes) advance by the offsets
                    const uint64_t at = ad0 + (uint64_t)((2 * tt * g.chunk_bytes) >> 4);
#pragma unroll
                    for (int kh = 0; kh < 9; ++kh) {
                        if (kh >= p.KH) break;
#pragma unroll
                        for (int s = 0; s < 2; ++s) {
                            if (s >= g.ksteps) break;
                            s_mma_lane0(d, at + (uint64_t)((2 * s * g.chunk_bytes + kh * 16) >> 4),
                                        bd0 + (uint64_t)(((kh * g.ksteps + s) * g.N * 32) >> 4),
                                        g.idesc, (kh | s) != 0, (uint32_t)lane);
                        }
                    }
                }
                s_commit_lane0(bar_full + 8u * tb, (uint32_t)lane);
            }
            s_commit_lane0(bar_free + 8u * ub, (uint32_t)lane);
        }
    } else {
        // ------------- weight staging and tensor-memory drain (warps 0-7) -------------
        // Channel c's banded matrices into weight buffer bsel: block
        // (kh, s) is an N x 16 K-major matrix whose row n = mm*16 + jj
        // holds at K = k the weight of output channel c*m + mm at kernel
        // column 16 s + k - a - jj (zero outside the kernel).
        auto stage_b = [&](int c, int bsel) {
            unsigned char *bsm = d_smem + g.b_off0 + bsel * g.b_bytes;
            const int rows = p.KH * g.ksteps * g.N;
            for (int row = t; row < rows; row += kDDrain) {
                const int blk = row / g.N;
                const int n = row - blk * g.N;
                const int kh = blk / g.ksteps, s = blk - kh * g.ksteps;
                const int mm = n >> 4, jj = n & 15;
                const T *wr = w + (int64_t)(c * g.m + mm) * p.ws[0] + (int64_t)kh * p.ws[2];
                unsigned char *dst = bsm + blk * g.N * 32 + (n >> 3) * 256 + (n & 7) * 16;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float v[8];
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        const int kw = 16 * s + 8 * h + cc - g.a - jj;
                        v[cc] = (kw >= 0 && kw < p.KW) ? load_f32(wr + (int64_t)kw * p.ws[3]) : 0.f;
                    }
                    uint4 o;
                    o.x = pack2(v[0], v[1], (T *)nullptr);
                    o.y = pack2(v[2], v[3], (T *)nullptr);
                    o.z = pack2(v[4], v[5], (T *)nullptr);
                    o.w = pack2(v[6], v[7], (T *)nullptr);
                    *reinterpret_cast<uint4 *>(dst + h * 128) = o;
                }
            }
        };
        int prev_c = -1, bsel = 1;
        // Before unit u (the k-th of this CTA): when its channel differs
        // from the previous unit's, its weights go to the other weight
        // buffer once the units that read that buffer (at least two back)
        // are through the tensor core; then every drain thread arrives on
        // b_ready of that buffer.
        auto stage = [&](const DtcUnit &u, int k) {
            if (u.c != prev_c) {
                prev_c = u.c;
                bsel ^= 1;
                if (k >= 2)
                    s_wait(bar_free + 8u * (uint32_t)((k - 2) % kDUnitBufs),
                           (uint32_t)(((k - 2) / kDUnitBufs) & 1), failed);
                stage_b(u.c, bsel);
                asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
                s_arrive(bar_bready + 8u * bsel);
            }
        };

        // Drain tile tt of unit u (global tile gt): warpgroup gt & 1 takes
        // it.  Thread r of the warpgroup holds output row 128 ot + r; it
        // reads the 16 columns of up to four output channels at once, frees
        // the tile buffer as soon as the last of them is in registers, adds
        // the bias, rounds once and stores 32 bytes per channel.
        const int qd = warp & 3, wg = warp >> 2;
        auto drain = [&](const DtcUnit &u, int tt, int gt) {
            const int tb = gt % g.bufs;
            const int r = 32 * qd + lane;
            const int oh = 128 * u.ot + r;
            const int ow0 = 16 * (g.owt * u.gw + tt);
            const bool row_ok = oh < p.OH && ow0 < p.OW;
            const uint32_t taddr = tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)(tb * g.N);
            for (int mb = 0; mb < g.m; mb += 4) {
                // the bias loads go out before the waits
                float bv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    bv[i] = (p.has_bias && mb + i < g.m)
                                ? load_f32(b + (int64_t)(u.c * g.m + mb + i) * p.bs)
                                : 0.f;
                if (mb == 0) {
                    s_wait(bar_full + 8u * tb, (uint32_t)((gt / g.bufs) & 1), failed);
                    s_fence_after();
                }
                float v[4][16];
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 4; ++i)   // the whole warp
                    if (mb + i < g.m) s_ld<16>(taddr + (uint32_t)(16 * (mb + i)), v[i]);
                s_wait_ld();
                if (mb + 4 >= g.m) {   // the tile buffer is read: free it
                    s_fence_before();
                    s_arrive(bar_empty + 8u * tb);
                }
                if (!row_ok) continue;
                const bool bad = *failed != 0;   // poison through the bias: NaN outputs
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (mb + i >= g.m) break;
                    const int co = u.c * g.m + mb + i;
                    const float bi = bad ? __int_as_float(0x7fc00000) : bv[i];
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[i][e] += bi;
                    T *yp = y + (int64_t)u.n * p.ys[0] + (int64_t)co * p.ys[1] +
                            (int64_t)oh * p.ys[2] + (int64_t)ow0 * p.ys[3];
                    if (g.vec_store && ow0 + 16 <= p.OW) {
                        uint32_t o[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            o[e] = pack2(v[i][2 * e], v[i][2 * e + 1], (T *)nullptr);
                        asm volatile(
                            "st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};\n" ::"l"(yp),
                            "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3]), "r"(o[4]), "r"(o[5]),
                            "r"(o[6]), "r"(o[7])
                            : "memory");
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            if (ow0 + e < p.OW) yp[(int64_t)e * p.ys[3]] = from_f32<T>(v[i][e]);
                    }
                }
            }
        };

        DtcUnit cur;
        cur.set(u0, g, p.N);
        int gt = 0;
        for (int k = 0; k < nunits; ++k) {
            stage(cur, k);
            for (int tt = 0; tt < g.owt; ++tt, ++gt)
                if ((gt & 1) == wg) drain(cur, tt, gt);
            cur.next(g, p.N);
        }
    }
    // Clean-up: the last unit's commits (and, after a failed wait, its
    // boxes) land before the shared and tensor memory go away.
    s_fence_before();
    __syncthreads();
    s_fence_after();
    if (t == 0) {
        const int kl = nunits - 1;
        if (*failed)
            for (int k = kl >= kDUnitBufs - 1 ? kl - (kDUnitBufs - 1) : 0; k <= kl; ++k)
                s_wait_final(bar_staged + 8u * (uint32_t)(k % kDUnitBufs),
                             (uint32_t)((k / kDUnitBufs) & 1));
        s_wait_final(bar_free + 8u * (uint32_t)(kl % kDUnitBufs), (uint32_t)((kl / kDUnitBufs) & 1));
    }
    __syncthreads();
    if (warp == kDWarps)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem),
                     "r"(g.tmem_cols));
}

template <typename T>
cudaError_t dwtc_launch_t(const Params &p, const Ptrs &q, cudaStream_t s, const DtcGeom &g) {
    // x as (W, H, C, N), column stride 1; boxes of 8 columns x R rows.
    CUtensorMap map;
    const uint64_t dims[4] = {(uint64_t)p.W, (uint64_t)p.H, (uint64_t)p.C_in, (uint64_t)p.N};
    const uint64_t strides[3] = {(uint64_t)p.xs[2] * sizeof(T), (uint64_t)p.xs[1] * sizeof(T),
                                 (uint64_t)p.xs[0] * sizeof(T)};
    const uint32_t box[4] = {8u, (uint32_t)g.R, 1u, 1u};
    if (!tma_encode_4d(&map, tma_dtype<T>(), q.x, dims, strides, box)) return cudaErrorInvalidValue;
    cudaError_t e =
        cudaFuncSetAttribute(dwtc_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem);
    if (e != cudaSuccess) return e;
    e = launch_kernel(dwtc_kernel<T>, dim3(g.ctas), dim3(kDThreads), g.smem, s, map,
                   static_cast<const T *>(q.w), static_cast<const T *>(q.b),
                   static_cast<T *>(q.y), p, g);
    return e != cudaSuccess ? e : cudaGetLastError();
}

bool dwtc_takes(const Params &p, const void *x) {
    // TMA boxes of 8 columns: 16-byte aligned base, column stride 1, row /
    // channel / image strides in whole 16-byte units.
    if (!aligned(x, 16)) return false;
    if (p.xs[3] != 1 || p.xs[2] % 8 || p.xs[1] % 8 || p.xs[0] % 8) return false;
    DtcGeom g;
    return dwtc_geometry(p, g);
}

bool dwtc_supports(const gconv_desc &d, const Ptrs &q) {
    return !d.transposed && dwtc_takes(make_params(d), q.x);
}

cudaError_t dwtc_launch(const Params &p, const Ptrs &q, cudaStream_t s, int *launches) {
    *launches = 1;
    DtcGeom g;
    if (!dwtc_geometry(p, g)) return cudaErrorNotSupported;
    // 32-byte stores of 16 output columns
    g.vec_store = aligned(q.y, 32) && p.ys[3] == 1 && p.ys[2] % 16 == 0 && p.ys[1] % 16 == 0 &&
                  p.ys[0] % 16 == 0;
    if (p.dtype == GCONV_BF16) return dwtc_launch_t<__nv_bfloat16>(p, q, s, g);
    return dwtc_launch_t<__half>(p, q, s, g);
}

}  // namespace

const Schedule kDwTc = {"dw_tc", dwtc_supports, dwtc_launch};

}  // namespace gconv
