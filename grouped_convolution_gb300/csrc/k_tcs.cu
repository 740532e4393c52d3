// k_tcs.cu -- grp_tc's shift form: few-channel grouped convolution at
// stride 2 (4 or 8 input channels per group, channels-last bf16/fp16) as an
// implicit GEMM on the tcgen05 tensor cores, with kernel columns in N.
//
// The convolution is the one of torch/_inductor/kernel/conv.py
// (LOOP_BODY_2D indexing, conv2d_template group offsets); executorch
// PR #25085 (description, second paragraph) leaves grouped convolutions
// whose per-group matrix product suits a tensor-core template to that
// template.  This form of the product is written for sm_103a:
//
//  - The unit of work is an 8-channel chunk (16 bytes per pixel: 8 / Cin_g
//    whole groups, NN = (8 / Cin_g) * Cout_g output channels) of Bo output
//    rows of one image.  The input is staged by four TMA boxes with a
//    traversal stride of 2 in both spatial dims: array (ph, s) holds, for
//    ring row i and entry e, the input pixel at row 2*(oh0 + i) - pad_h + s
//    and column 2*(ow0 + e) - cpad + ph (cpad = pad_w rounded up to even),
//    zero outside the image: its rows back to back, one 16-byte entry per
//    pixel.
//  - With tap kw + (cpad - pad_w) = 2j + ph, output column p reads entry
//    p + j of phase ph.  A row r (the MMA's M = 128 rows) is one entry; the
//    two K halves of an MMA (K = 16) are that entry's two phases, arrays
//    (0, s) and (1, s) (the descriptor's leading byte offset is the distance
//    between them); N holds the NN output channels of each column shift j
//    (N = J * NN).  Per kernel row kh there is one MMA (arrays (ph, kh & 1),
//    ring row offset kh >> 1):
//      D[r][j*NN + n] += sum_{ph, c} A_ph[r][c] * w[n, c, kh, 2j + ph - dc]
//    (dc = cpad - pad_w; zero weights outside the kernel or n's group).
//    Output column p is the sum over j of D[p + j][j*NN + n]: the J
//    accumulator blocks of a row are read once from tensor memory and the
//    shifted ones added with warp shuffles.  Each staged entry is read by
//    the tensor core once per kernel row instead of once per tap.
//  - Entries of consecutive output rows follow each other in the arrays
//    (ring row i + 1 is the next output row), so a tile is 128 consecutive
//    entries of the band, whichever rows they belong to; tiles advance by
//    TS = 128 - (J - 1) entries so every output finds its shifted rows in
//    one tile.  Row entries E = OWt + J - 1 per output row.
//  - One CTA per SM: eight warps stage (all stage the chunk's weights when
//    the chunk changes) and drain tensor memory, the two warpgroups taking
//    alternate tiles; one warp issues the input boxes and three warps issue
//    the MMAs of every third tile (one warp issues an MMA every ~74 cycles
//    at best, the tensor core takes one of N = 80 every ~52 cycles).  Two
//    unit buffers and six tensor-memory tile buffers keep the tensor core
//    fed while the next unit is staged and earlier tiles are drained.
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

constexpr int kSWarps = 16;                  // staging + drain
constexpr int kSProducers = 32 * kSWarps;
constexpr int kSDrainGroups = kSWarps / 4;   // warpgroups that drain tiles in turn
constexpr int kSIssuers = 3;                 // MMA issue warps
constexpr int kSLoader = kSWarps + kSIssuers;   // the warp that issues the input boxes
constexpr int kSThreads = kSProducers + 32 * (kSIssuers + 1);
constexpr int kSMaxJ = 5;                    // column shifts (KW <= 9)
constexpr int kSTileBufs = 6;                // tensor-memory tile buffers (N <= 80: 480 columns)
constexpr int kSSmemCap = 220 * 1024;
// Exchange rows between the warps of a warpgroup: [warpgroup][tile parity]
// [warp][lane < 4][(j - 1) * NN + c], lanes kSLane floats apart so the four
// writers (and readers) of a 16-byte vector hit different banks.
template <int NNT> constexpr int kSLane = (kSMaxJ - 1) * NNT + 4;
constexpr int kSXchFloats = kSDrainGroups * 2 * 4 * 4 * kSLane<16>;

struct TcsGeom {
    int NN, J, N;          // chunk outputs, column shifts, MMA N (16 | N)
    int dc, cpad;          // cpad - pad_w (0 or 1), pad_w rounded up to even
    int Bo, OWt, E, TS, Tn, R, R_load, Lv;
    int chunks, bands, cts, units, ctas;
    int arr_bytes;         // one (ph, s) array, 128-byte aligned
    int ring_bytes;        // the four arrays of one unit buffer
    int b_bytes;           // one weight buffer (KH blocks)
    int raw_elems;         // the chunk's weights: NN x Cin_g x KH x KW
    int w_dense;           // weights dense and 16-byte aligned per chunk
    int ring_off[2], b_off[2], x_off, bias_off, bar_off, smem;
    int tmem_cols;
    uint32_t idesc;
    FastDiv Ediv, Ndiv;
    int nn_shift, cout_shift;   // log2(NN), log2(Cout_g)
    int vec_store;         // 0: element stores, 1: 16-byte, 2: 32-byte vectors
};

bool tcs_geometry(const Params &p, TcsGeom &g) {
    if (p.sh != 2 || p.sw != 2 || p.dh != 1 || p.dw != 1 || p.transposed) return false;
    if (p.Cin_g != 4 && p.Cin_g != 8) return false;
    if (p.C_in % 8 != 0) return false;
    if (p.KH < 1 || p.KH > 9 || p.KW < 1 || p.KW > 9) return false;
    g.NN = (8 / p.Cin_g) * p.Cout_g;
    if (g.NN != 8 && g.NN != 16) return false;
    g.nn_shift = g.NN == 8 ? 3 : 4;
    g.cout_shift = 0;
    while ((1 << g.cout_shift) < p.Cout_g) ++g.cout_shift;   // Cout_g = NN * Cin_g / 8: 4, 8 or 16
    g.dc = p.pbw & 1;
    g.cpad = p.pbw + g.dc;
    g.J = (p.KW + g.dc + 1) / 2;
    if (g.J > kSMaxJ) return false;
    g.N = (g.J * g.NN + 15) / 16 * 16;
    g.TS = 128 - (g.J - 1);
    // Column tiles of at most 120 outputs; rows per unit as many (<= 8) as fit.
    g.cts = (p.OW + 119) / 120;
    g.OWt = (p.OW + g.cts - 1) / g.cts;
    g.E = g.OWt + g.J - 1;   // an output's last shift reads entry p + J - 1
    g.b_bytes = (p.KH * g.N * 32 + 127) / 128 * 128;
    g.raw_elems = g.NN * p.Cin_g * p.KH * p.KW;
    const int x_bytes = (g.raw_elems * 2 > kSXchFloats * 4 ? g.raw_elems * 2 : kSXchFloats * 4);
    const int fixed = 2 * g.b_bytes + (x_bytes + 127) / 128 * 128 + 2 * 16 * 4 + 256;
    g.Bo = 0;
    for (int bo = (p.OH < 8 ? p.OH : 8); bo >= 1; --bo) {
        const int Lv = (bo - 1) * g.E + g.OWt;
        const int Tn = (Lv + g.TS - 1) / g.TS;
        const int maxe = ((p.KH - 1) / 2) * g.E + (Tn - 1) * g.TS + 128;
        const int R = maxe / g.E + 1;
        if (2 * R > 256 || 2 * g.E > 256) continue;   // TMA box extents
        const int arr = (R * g.E * 16 + 127) / 128 * 128;
        if (2 * 4 * arr + fixed > kSSmemCap) continue;
        g.Bo = bo;
        g.Lv = Lv;
        g.Tn = Tn;
        g.R = R;
        g.arr_bytes = arr;
        break;
    }
    if (g.Bo == 0) return false;
    // Rows past Bo + (KH - 1) / 2 are read only by accumulator rows that no
    // output uses (the last tile's overrun), so they are not loaded.
    g.R_load = g.Bo + (p.KH - 1) / 2;
    g.ring_bytes = 4 * g.arr_bytes;
    g.chunks = p.C_in / 8;
    g.bands = (p.OH + g.Bo - 1) / g.Bo;
    const int64_t units = (int64_t)g.chunks * p.N * g.bands * g.cts;
    if (units > INT32_MAX) return false;
    g.units = (int)units;
    g.ctas = g.units < 152 ? g.units : 152;
    g.ring_off[0] = 0;
    g.ring_off[1] = g.ring_bytes;
    g.b_off[0] = 2 * g.ring_bytes;
    g.b_off[1] = g.b_off[0] + g.b_bytes;
    g.x_off = g.b_off[1] + g.b_bytes;
    g.bias_off = g.x_off + (x_bytes + 127) / 128 * 128;
    g.bar_off = g.bias_off + 2 * 16 * 4;
    g.smem = g.bar_off + 32 + 16 * kSTileBufs + 32;
    if (g.smem > kSSmemCap) return false;
    int cols = kSTileBufs * g.N, pow2 = 32;
    while (pow2 < cols) pow2 *= 2;
    if (pow2 > 512) return false;
    g.tmem_cols = pow2;
    g.idesc = s_idesc(p.dtype == GCONV_BF16, 128, g.N);
    g.Ediv = FastDiv((uint32_t)g.E);
    g.Ndiv = FastDiv((uint32_t)g.N);
    g.w_dense = 0;
    g.vec_store = 0;
    return true;
}

// Division-free cursor over units (column tile fastest, then band, image,
// chunk): consecutive units of a CTA share the chunk's weights.
struct TcsUnit {
    int c, n, b, ct;
    __device__ __forceinline__ void set(int u, const TcsGeom &g, int N) {
        ct = u % g.cts;
        int r = u / g.cts;
        b = r % g.bands;
        r /= g.bands;
        n = r % N;
        c = r / N;
    }
    __device__ __forceinline__ void next(const TcsGeom &g, int N) {
        if (++ct < g.cts) return;
        ct = 0;
        if (++b < g.bands) return;
        b = 0;
        if (++n < N) return;
        n = 0;
        ++c;
    }
};

__device__ __forceinline__ void s_producer_sync() {   // warps 0-7 only
    asm volatile("bar.sync 1, %0;\n" ::"n"(kSProducers) : "memory");
}
__device__ __forceinline__ void s_group_sync(int wg) {  // warps 4wg .. 4wg+3
    asm volatile("bar.sync %0, 128;\n" ::"r"(2 + wg) : "memory");
}

// T: element type; NNT: output channels per chunk (8 or 16).
template <typename T, int NNT>
__global__ void __launch_bounds__(kSThreads, 1)
tcs_kernel(const __grid_constant__ CUtensorMap xmap, const T *__restrict__ w,
           const T *__restrict__ b, T *__restrict__ y, Params p, TcsGeom g) {
    pdl_launch_dependents();
    pdl_wait();
    extern __shared__ __align__(1024) unsigned char s_smem[];
    const uint32_t sbase = smem_addr(s_smem);
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int per = g.units / g.ctas, extra = g.units % g.ctas;
    const int u0 = blockIdx.x * per + min((int)blockIdx.x, extra);
    const int nunits = per + ((int)blockIdx.x < extra ? 1 : 0);
    if (nunits <= 0) return;

    // mbarriers: staged[2] (a unit's four boxes landed: the loader's
    // expect-tx arrival), ring_free[2] (every MMA that read the unit buffer
    // completed: one commit per issuer), acc_full[4] (a tile's MMAs
    // completed), acc_empty[4] (a tile drained by its warpgroup: 128
    // arrivals), b_ready[2] (a chunk's weights and bias written into weight
    // buffer i: 256 arrivals).
    const uint32_t bar_staged = sbase + (uint32_t)g.bar_off;
    const uint32_t bar_free = bar_staged + 16u;
    const uint32_t bar_full = bar_staged + 32u;
    const uint32_t bar_empty = bar_full + 8u * kSTileBufs;
    const uint32_t bar_bready = bar_empty + 8u * kSTileBufs;
    constexpr int kSlot = 32 + 16 * kSTileBufs + 16;   // byte offset of the TMEM address slot
    uint32_t *tslot = reinterpret_cast<uint32_t *>(s_smem + g.bar_off + kSlot);
    volatile int *failed = reinterpret_cast<volatile int *>(s_smem + g.bar_off + kSlot + 4);
    float *bias_s = reinterpret_cast<float *>(s_smem + g.bias_off);   // [2][16]
    float *xch = reinterpret_cast<float *>(s_smem + g.x_off);

    if (warp == kSWarps) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                         sbase + (uint32_t)(g.bar_off + kSlot)),
                     "r"(g.tmem_cols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
    }
    if (t == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_staged + 8u * i, 1);
            mbar_init(bar_free + 8u * i, kSIssuers);
            mbar_init(bar_bready + 8u * i, kSProducers);
        }
        for (int i = 0; i < kSTileBufs; ++i) {
            mbar_init(bar_full + 8u * i, 1);
            mbar_init(bar_empty + 8u * i, kSProducers / kSDrainGroups);
        }
        *failed = 0;
        fence_barrier_init();
        tma_prefetch_map(&xmap);
    }
    s_fence_before();
    __syncthreads();
    s_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == kSLoader) {
        // ------ input boxes: unit k into unit buffer k & 1 once the tensor
        // core has read the unit two back ------
        // The whole warp runs the loop; lane 0 issues.
        const uint32_t box_bytes = (uint32_t)(16 * g.E * g.R_load);
        TcsUnit u;
        u.set(u0, g, p.N);
        for (int k = 0; k < nunits; ++k, u.next(g, p.N)) {
            const int ub = k & 1;
            if (k >= 2) s_wait_warp(bar_free + 8u * ub, (uint32_t)(((k - 2) >> 1) & 1), failed);
            s_expect_tx_lane0(bar_staged + 8u * ub, 4u * box_bytes, (uint32_t)lane);
            const int oh0 = u.b * g.Bo, ow0 = u.ct * g.OWt;
            const uint32_t ring = sbase + (uint32_t)g.ring_off[ub];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int ph = a >> 1, s = a & 1;
                s_tma_lane0(ring + (uint32_t)((ph * 2 + s) * g.arr_bytes), &xmap,
                            bar_staged + 8u * ub, 8 * u.c, 2 * ow0 - g.cpad + ph,
                            2 * oh0 - p.pbh + s, u.n, (uint32_t)lane);
            }
        }
    } else if (warp >= kSWarps) {
        // ------ MMA issue: issuer i takes tiles i, i+3, ...; the whole warp
        // runs the loop (warp-uniform descriptors), lane 0 issues ------
        const int iss = warp - kSWarps;
        int gt = 0;
        TcsUnit u;
        u.set(u0, g, p.N);
        int prev_c = -1, bsel = 1, bstaged = 0;   // bit i: phase of b_ready[i]
        for (int k = 0; k < nunits; ++k, u.next(g, p.N)) {
            const int ub = k & 1;
            if (u.c != prev_c) {   // the weights of a new chunk, in the other buffer
                prev_c = u.c;
                bsel ^= 1;
                s_wait_warp(bar_bready + 8u * bsel, (uint32_t)((bstaged >> bsel) & 1), failed);
                bstaged ^= 1 << bsel;
            }
            s_wait_warp(bar_staged + 8u * ub, (uint32_t)((k >> 1) & 1), failed);
            s_fence_after();
            // Descriptors of kh's operands for tile 0: A from array (0, kh & 1)
            // at ring row kh >> 1, its second K half (phase 1) in array
            // (1, kh & 1), two arrays on (leading byte offset); tile tt adds
            // tt * TS entries to A's start address, the descriptor's low field
            // in 16-byte units (no carry: shared addresses stay below 2^18).
            const uint32_t ring = sbase + (uint32_t)g.ring_off[ub];
            uint64_t ad0[9];
#pragma unroll
            for (int kh = 0; kh < 9; ++kh)
                ad0[kh] = s_desc(ring + (uint32_t)((kh & 1) * g.arr_bytes) +
                                     (uint32_t)((kh >> 1) * g.E * 16),
                                 (uint32_t)(2 * g.arr_bytes), 128);
            const uint64_t bd0 = s_desc(sbase + (uint32_t)g.b_off[bsel], 128, 256);
            const uint64_t bstep = (uint64_t)(g.N * 32 / 16);
            for (int tt = 0; tt < g.Tn; ++tt, ++gt) {
                if (gt % kSIssuers != iss) continue;
                const int tb = gt % kSTileBufs;
                const int use = gt / kSTileBufs;
                if (use >= 1) s_wait_warp(bar_empty + 8u * tb, (uint32_t)((use - 1) & 1), failed);
                s_fence_after();
                if (!__any_sync(0xffffffffu, *failed != 0)) {
                    const uint32_t d = tmem + (uint32_t)(tb * g.N);
                    const uint64_t toff = (uint64_t)(tt * g.TS);
#pragma unroll
                    for (int kh = 0; kh < 9; ++kh)
                        if (kh < p.KH)
                            s_mma_lane0(d, ad0[kh] + toff, bd0 + (uint64_t)kh * bstep, g.idesc,
                                        kh, (uint32_t)lane);
                }
                s_commit_lane0(bar_full + 8u * tb, (uint32_t)lane);
            }
            s_commit_lane0(bar_free + 8u * ub, (uint32_t)lane);
        }
    } else {
        // ------------- staging and tensor-memory drain (warps 0-7) -------------
        // Chunk c's weights into weight buffer bsel.  First the chunk's raw
        // weights [NN][Cin_g][KH][KW] into shared memory (16-byte loads when
        // they are dense and aligned), then the operand: block kh is an
        // N x 16 K-major matrix whose row n = j*NN + n' (output channel
        // c*NN + n') holds at K = ph*8 + cc the weight of chunk channel cc at
        // kernel column 2j + ph - dc, zero outside the kernel and outside
        // n''s group.  The raw copy shares the exchange buffer
        // (every producer is inside stage() here).
        auto stage_b = [&](int c, int bsel) {
            T *raw = reinterpret_cast<T *>(xch);
            if (g.w_dense) {
                // at most 16 x 8 x 81 / 8 = 1296 vectors, all of a thread's
                // loads in flight before its stores
                const uint4 *src = reinterpret_cast<const uint4 *>(w + (int64_t)c * g.raw_elems);
                constexpr int kV = (1296 + kSProducers - 1) / kSProducers;
                uint4 v[kV];
#pragma unroll
                for (int i = 0; i < kV; ++i) {
                    const int e = t + i * kSProducers;
                    v[i] = e < g.raw_elems / 8 ? __ldg(src + e) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int i = 0; i < kV; ++i) {
                    const int e = t + i * kSProducers;
                    if (e < g.raw_elems / 8) reinterpret_cast<uint4 *>(raw)[e] = v[i];
                }
            } else {
                const int khw = p.KH * p.KW;
                for (int e = t; e < g.raw_elems; e += kSProducers) {
                    const int np = e / (p.Cin_g * khw);
                    const int r1 = e - np * p.Cin_g * khw;
                    const int ci = r1 / khw, r2 = r1 - ci * khw;
                    const int kh = r2 / p.KW, kw = r2 - kh * p.KW;
                    raw[e] = w[(int64_t)(c * g.NN + np) * p.ws[0] + (int64_t)ci * p.ws[1] +
                               (int64_t)kh * p.ws[2] + (int64_t)kw * p.ws[3]];
                }
            }
            s_producer_sync();
            unsigned char *bsm = s_smem + g.b_off[bsel];
            const int rows = p.KH * g.N;
            for (int row = t; row < rows; row += kSProducers) {
                const int kh = (int)g.Ndiv.div((uint32_t)row);
                const int n = row - kh * g.N;
                const int j = n >> g.nn_shift, np = n & (g.NN - 1);
                const int cb = (np >> g.cout_shift) * p.Cin_g;
                unsigned char *dst = bsm + kh * g.N * 32 + (n >> 3) * 256 + (n & 7) * 16;
#pragma unroll
                for (int ph = 0; ph < 2; ++ph) {
                    const int kw = 2 * j + ph - g.dc;
                    const bool kw_ok = j < g.J && kw >= 0 && kw < p.KW;
                    float v[8];
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        const bool ok = kw_ok && cc >= cb && cc < cb + p.Cin_g;
                        const int ri = ok ? ((np * p.Cin_g + cc - cb) * p.KH + kh) * p.KW + kw : 0;
                        const float f = Elem<T>::to_f32(raw[ri]);
                        v[cc] = ok ? f : 0.f;
                    }
                    uint4 o;
                    o.x = pack2(v[0], v[1], (T *)nullptr);
                    o.y = pack2(v[2], v[3], (T *)nullptr);
                    o.z = pack2(v[4], v[5], (T *)nullptr);
                    o.w = pack2(v[6], v[7], (T *)nullptr);
                    *reinterpret_cast<uint4 *>(dst + ph * 128) = o;
                }
            }
        };
        int prev_c = -1, bsel = 1;
        int ubsel_bits = 0;   // bit ub: the weight buffer of the unit in unit buffer ub
        // Before unit u (the k-th of this CTA): when its chunk differs from
        // the previous unit's, its weights and bias go to the other weight
        // buffer once the units that read that buffer (at least two back)
        // are through the tensor core; then every producer arrives on
        // b_ready of that buffer.
        auto stage = [&](const TcsUnit &u, int k) {
            const int ub = k & 1;
            if (u.c != prev_c) {
                prev_c = u.c;
                bsel ^= 1;
                // every producer is done with the exchange buffer (the raw
                // weights go there) and with the bias of two chunks back
                s_producer_sync();
                if (k >= 2) s_wait(bar_free + 8u * ub, (uint32_t)(((k - 2) >> 1) & 1), failed);
                stage_b(u.c, bsel);
                if (t < g.NN)
                    bias_s[bsel * 16 + t] =
                        p.has_bias ? load_f32(b + (int64_t)(u.c * g.NN + t) * p.bs) : 0.f;
                asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
                s_producer_sync();   // the raw copy in the exchange buffer is done with
                s_arrive(bar_bready + 8u * bsel);
            }
            ubsel_bits = (ubsel_bits & ~(1 << ub)) | (bsel << ub);
        };

        // Drain tile tt of unit u (global tile gt): warpgroup gt % 4 takes
        // it (the warpgroups drain tiles in turn).  Warp qd reads its 32
        // accumulator rows two column blocks at a time and adds block j of
        // the row j below (a shuffle inside the warp); lanes 0..J-2 leave
        // their blocks for the warp above, whose last lanes add them after
        // the warpgroup's barrier.  Then the bias, one rounding and 2 * NN
        // bytes stored per output pixel.
        const int qd = warp & 3, wg = warp >> 2;
        auto drain = [&](const TcsUnit &u, int k, int tt, int gt) {
            const int ub = k & 1;
            const int tb = gt % kSTileBufs;
            s_wait(bar_full + 8u * tb, (uint32_t)((gt / kSTileBufs) & 1), failed);
            s_fence_after();
            const uint32_t taddr = tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)(tb * g.N);
            constexpr int kLane = kSLane<NNT>;
            constexpr int kXW = 4 * kLane;   // floats per warp
            float *xw = xch + ((wg * 2 + ((gt / kSDrainGroups) & 1)) * 4 + qd) * kXW;
            float acc[NNT];
#pragma unroll
            for (int j0 = 0; j0 < kSMaxJ; j0 += 2) {
                if (j0 >= g.J) break;
                float blk[2][NNT];
                s_ld<NNT>(taddr + (uint32_t)(j0 * NNT), blk[0]);
                if (j0 + 1 < g.J) s_ld<NNT>(taddr + (uint32_t)((j0 + 1) * NNT), blk[1]);
                s_wait_ld();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int j = j0 + h;
                    if (j >= g.J || j >= kSMaxJ) break;
                    if (j == 0) {
#pragma unroll
                        for (int c = 0; c < NNT; ++c) acc[c] = blk[0][c];
                        continue;
                    }
                    // row m < j of this warp is read at shift j by row
                    // m - j + 32 of the warp above
                    if (lane < j) {
#pragma unroll
                        for (int c4 = 0; c4 < NNT / 4; ++c4)
                            *reinterpret_cast<float4 *>(xw + lane * kLane + (j - 1) * NNT + 4 * c4) =
                                make_float4(blk[h][4 * c4], blk[h][4 * c4 + 1], blk[h][4 * c4 + 2],
                                            blk[h][4 * c4 + 3]);
                    }
                    const bool inside = lane + j < 32;
#pragma unroll
                    for (int c = 0; c < NNT; ++c) {
                        const float v = __shfl_down_sync(0xffffffffu, blk[h][c], j);
                        acc[c] += inside ? v : 0.f;
                    }
                }
            }
            s_fence_before();
            s_arrive(bar_empty + 8u * tb);
            s_group_sync(wg);
            // the last lanes: rows of the next warp (none past the tile)
            if (qd < 3 && lane + g.J - 1 >= 32) {
                const float *xn = xw + kXW;   // the next warp of the group (qd + 1)
#pragma unroll
                for (int j = 1; j < kSMaxJ; ++j) {
                    if (j >= g.J) break;
                    if (lane + j < 32) continue;
                    const int m = lane + j - 32;
#pragma unroll
                    for (int c4 = 0; c4 < NNT / 4; ++c4) {
                        const float4 v =
                            *reinterpret_cast<const float4 *>(xn + m * kLane + (j - 1) * NNT + 4 * c4);
                        acc[4 * c4] += v.x;
                        acc[4 * c4 + 1] += v.y;
                        acc[4 * c4 + 2] += v.z;
                        acc[4 * c4 + 3] += v.w;
                    }
                }
            }
            const int r = 32 * qd + lane;
            const int vpos = tt * g.TS + r;
            const int q = (int)g.Ediv.div((uint32_t)vpos);
            const int pc = vpos - q * g.E;
            const int oh = u.b * g.Bo + q, ow = u.ct * g.OWt + pc;
            const bool ok = r < g.TS && vpos < g.Lv && pc < g.OWt && q < g.Bo && oh < p.OH &&
                            ow < p.OW;
            if (!ok) return;
            const float *bs = bias_s + ((ubsel_bits >> ub) & 1) * 16;
            float f[NNT];
#pragma unroll
            for (int c = 0; c < NNT; ++c) f[c] = acc[c] + bs[c];
            if (*failed != 0) {   // a failed CTA writes NaN
#pragma unroll
                for (int c = 0; c < NNT; ++c) f[c] = __int_as_float(0x7fc00000);
            }
            const int co0 = u.c * NNT;
            T *yp = y + (int64_t)u.n * p.ys[0] + (int64_t)oh * p.ys[2] + (int64_t)ow * p.ys[3] +
                    (int64_t)co0 * p.ys[1];
            if (NNT == 16 && g.vec_store == 2) {
                // one 32-byte store: the pixel's whole sector
                uint32_t o[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) o[i] = pack2(f[2 * i], f[2 * i + 1], (T *)nullptr);
                asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};\n" ::"l"(yp),
                             "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3]), "r"(o[4]), "r"(o[5]),
                             "r"(o[6]), "r"(o[7])
                             : "memory");
            } else if (g.vec_store) {
#pragma unroll
                for (int v8 = 0; v8 < NNT / 8; ++v8) {
                    uint4 o;
                    o.x = pack2(f[8 * v8 + 0], f[8 * v8 + 1], (T *)nullptr);
                    o.y = pack2(f[8 * v8 + 2], f[8 * v8 + 3], (T *)nullptr);
                    o.z = pack2(f[8 * v8 + 4], f[8 * v8 + 5], (T *)nullptr);
                    o.w = pack2(f[8 * v8 + 6], f[8 * v8 + 7], (T *)nullptr);
                    reinterpret_cast<uint4 *>(yp)[v8] = o;
                }
            } else {
#pragma unroll
                for (int c = 0; c < NNT; ++c) yp[(int64_t)c * p.ys[1]] = from_f32<T>(f[c]);
            }
        };

        TcsUnit cur;
        cur.set(u0, g, p.N);
        TcsUnit nxt = cur;
        nxt.next(g, p.N);
        stage(cur, 0);
        int gt = 0;
        for (int k = 0; k < nunits; ++k) {
            if (k + 1 < nunits) stage(nxt, k + 1);
            for (int tt = 0; tt < g.Tn; ++tt, ++gt)
                if (gt % kSDrainGroups == wg) drain(cur, k, tt, gt);
            cur = nxt;
            nxt.next(g, p.N);
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
            for (int k = kl > 0 ? kl - 1 : 0; k <= kl; ++k)
                s_wait_final(bar_staged + 8u * (uint32_t)(k & 1), (uint32_t)((k >> 1) & 1));
        s_wait_final(bar_free + 8u * (uint32_t)(kl & 1), (uint32_t)((kl >> 1) & 1));
    }
    __syncthreads();
    if (warp == kSWarps)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem),
                     "r"(g.tmem_cols));
}

template <typename T>
cudaError_t tcs_launch_t(const Params &p, const Ptrs &q, cudaStream_t s, const TcsGeom &g) {
    // x as (C_in, W, H, N), channel stride 1; boxes of 8 channels x E pixels
    // (every second column) x R rows (every second row).
    CUtensorMap map;
    const uint64_t dims[4] = {(uint64_t)p.C_in, (uint64_t)p.W, (uint64_t)p.H, (uint64_t)p.N};
    const uint64_t strides[3] = {(uint64_t)p.xs[3] * sizeof(T), (uint64_t)p.xs[2] * sizeof(T),
                                 (uint64_t)p.xs[0] * sizeof(T)};
    const uint32_t box[4] = {8u, (uint32_t)(2 * g.E), (uint32_t)(2 * g.R_load), 1u};
    const uint32_t estr[4] = {1u, 2u, 2u, 1u};
    if (!tma_encode_4d_strided(&map, tma_dtype<T>(), q.x, dims, strides, box, estr))
        return cudaErrorInvalidValue;
    cudaError_t e;
    if (g.NN == 16) {
        e = cudaFuncSetAttribute(tcs_kernel<T, 16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 g.smem);
        if (e != cudaSuccess) return e;
        e = launch_kernel(tcs_kernel<T, 16>, dim3(g.ctas), dim3(kSThreads), g.smem, s, map,
                       static_cast<const T *>(q.w), static_cast<const T *>(q.b),
                       static_cast<T *>(q.y), p, g);
    } else {
        e = cudaFuncSetAttribute(tcs_kernel<T, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 g.smem);
        if (e != cudaSuccess) return e;
        e = launch_kernel(tcs_kernel<T, 8>, dim3(g.ctas), dim3(kSThreads), g.smem, s, map,
                       static_cast<const T *>(q.w), static_cast<const T *>(q.b),
                       static_cast<T *>(q.y), p, g);
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

bool tcs_takes(const Params &p, const void *x) {
    if (p.layout != GCONV_LAYOUT_NHWC) return false;
    if (p.dtype != GCONV_BF16 && p.dtype != GCONV_F16) return false;
    // TMA boxes of 8 channels: 16-byte aligned base, channel stride 1,
    // pixel / row / image strides in whole 8-channel units.
    if (!aligned(x, 16)) return false;
    if (p.xs[1] != 1 || p.xs[3] % 8 || p.xs[2] % 8 || p.xs[0] % 8) return false;
    TcsGeom g;
    return tcs_geometry(p, g);
}

bool tcs_supports(const gconv_desc &d, const Ptrs &q) {
    return plain_forward(d) && tcs_takes(make_params(d), q.x);
}

cudaError_t tcs_launch(const Params &p, const Ptrs &q, cudaStream_t s, int *launches) {
    *launches = 1;
    TcsGeom g;
    if (!tcs_geometry(p, g)) return cudaErrorNotSupported;
    // the chunk's weights as one dense run of 16-byte vectors
    g.w_dense = p.ws[3] == 1 && p.ws[2] == p.KW && p.ws[1] == (int64_t)p.KH * p.KW &&
                p.ws[0] == (int64_t)p.Cin_g * p.KH * p.KW && g.raw_elems % 8 == 0 &&
                aligned(q.w, 16);
    // 16-byte stores of 8 output channels
    g.vec_store = aligned(q.y, 16) && p.ys[1] == 1 && p.ys[3] % 8 == 0 && p.ys[2] % 8 == 0 &&
                  p.ys[0] % 8 == 0;
    // 32-byte stores of 16 output channels
    if (g.vec_store && g.NN == 16 && aligned(q.y, 32) && p.ys[3] % 16 == 0 &&
        p.ys[2] % 16 == 0 && p.ys[0] % 16 == 0)
        g.vec_store = 2;
    if (p.dtype == GCONV_BF16) return tcs_launch_t<__nv_bfloat16>(p, q, s, g);
    return tcs_launch_t<__half>(p, q, s, g);
}

}  // namespace gconv
