// k_tcs.cu -- grp_tc's shift form: few-channel grouped convolution at
// stride 2 (4 or 8 input channels per group, channels-last bf16/fp16) as an
// implicit GEMM on the tcgen05 tensor cores, with the kernel columns in N.
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
//    zero outside the image.  Each array is its rows back to back, one
//    16-byte entry per pixel.
//  - With tap kw + (cpad - pad_w) = 2j + ph, output column p of the tile
//    reads entry p + j.  So A row r (the MMA's M = 128 rows) is one entry,
//    the two K halves of an MMA (K = 16) are the ph = 0 and ph = 1 entries
//    of one kernel row kh (s = kh & 1, ring row offset kh >> 1), and N
//    holds the NN output channels for each of the J column shifts j:
//      D[r][j*NN + n] = sum_{kh, ph, c} A_{kh}[r][ph, c] * w[n, c, kh, 2j + ph - dc]
//    (dc = cpad - pad_w; zero weights outside the kernel or n's group).
//    The output pixel p is the sum over j of D[p + j][j*NN + n]: each
//    accumulator row is read once from tensor memory and the shifts are
//    added with warp shuffles.  One MMA covers J kernel columns, so every
//    staged entry is read by the tensor core once per kernel row instead of
//    once per tap.
//  - Entries of consecutive output rows follow each other in the arrays
//    (ring row i + 1 is the next output row), so a tile is 128 consecutive
//    entries of the band, whichever rows they belong to; tiles advance by
//    TS = 128 - (J - 1) entries so every output finds its J shifted rows
//    in one tile.  Row entries E = OWt + J - 1 per output row.
//  - One CTA per SM: eight warps stage (one thread issues the TMA boxes;
//    all stage the chunk's weights when the chunk changes) and drain tensor
//    memory; two warps issue the MMAs of alternate tiles.  Two unit buffers
//    and four tensor-memory tile buffers keep the tensor core fed while the
//    next unit is staged and the previous tiles are drained.
//  - Every mbarrier wait is bounded; a wait that gives up marks the CTA
//    failed, its outputs are written as NaN, and before exiting the CTA
//    waits (bounded) for its copies and MMAs in flight before it frees its
//    tensor memory.
#include <cstdint>

#include "device_common.cuh"
#include "gconv_internal.h"
#include "launch.cuh"
#include "tma.cuh"

namespace gconv {
namespace {

constexpr int kSWarps = 8;                   // staging + drain
constexpr int kSProducers = 32 * kSWarps;
constexpr int kSIssuers = 2;                 // MMA issue warps
constexpr int kSThreads = kSProducers + 32 * kSIssuers;
constexpr int kSMaxJ = 5;                    // column shifts (KW <= 9)
constexpr int kSMaxHalf = 8;                 // output channels per drain warp
constexpr int kSTileBufs = 4;
constexpr int kSSmemCap = 220 * 1024;
constexpr uint32_t kSSpinLimit = 1u << 22;

struct TcsGeom {
    int NN, J, N;          // chunk outputs, column shifts, MMA N (16 | N)
    int dc;                // cpad - pad_w (0 or 1)
    int cpad;
    int Bo, OWt, E, TS, Tn, R, Lv;
    int chunks, bands, cts, units, ctas;
    int arr_bytes;         // one (ph, s) array, 128-byte aligned
    int ring_bytes;        // the four arrays of one unit buffer
    int b_bytes;           // one weight buffer (KH slices)
    int ring_off[2], b_off[2], x_off, bias_off, bar_off, smem;
    int tmem_cols;
    uint32_t idesc;
    FastDiv Ediv;
    int vec_store;
};

// 64-bit shared-memory matrix descriptor (tcgen05): K-major, no swizzle;
// start address, leading byte offset (between the two K-adjacent 8x16-byte
// core matrices), stride byte offset (between M/N-adjacent ones), in 16-byte
// units; bit 46 holds the descriptor version.
__device__ __forceinline__ uint64_t s_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo & 0x3FFFFu) >> 4) << 16) |
           ((uint64_t)((sbo & 0x3FFFFu) >> 4) << 32) | ((uint64_t)1 << 46);
}

// kind::f16 instruction descriptor: fp32 accumulator, A and B both bf16 or
// both fp16, both K-major, N / 8 and M / 16.
inline uint32_t s_idesc(bool bf16, int M, int N) {
    const uint32_t ab = bf16 ? 1u : 0u;
    return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

bool tcs_geometry(const Params &p, TcsGeom &g) {
    if (p.sh != 2 || p.sw != 2 || p.dh != 1 || p.dw != 1 || p.transposed) return false;
    if (p.Cin_g != 4 && p.Cin_g != 8) return false;
    if (p.C_in % 8 != 0) return false;
    if (p.KH < 1 || p.KH > 9 || p.KW < 1 || p.KW > 9) return false;
    g.NN = (8 / p.Cin_g) * p.Cout_g;
    if (g.NN != 8 && g.NN != 16) return false;
    g.dc = p.pbw & 1;
    g.cpad = p.pbw + g.dc;
    g.J = (p.KW + g.dc + 1) / 2;
    if (g.J > kSMaxJ) return false;
    g.N = (g.J * g.NN + 15) / 16 * 16;
    if (g.N > 256) return false;
    g.TS = 128 - (g.J - 1);
    // Column tiles of at most 120 outputs; rows per unit as many (<= 8) as fit.
    g.cts = (p.OW + 119) / 120;
    g.OWt = (p.OW + g.cts - 1) / g.cts;
    g.E = g.OWt + g.J - 1;
    const int b_bytes = p.KH * g.N * 32;
    g.b_bytes = (b_bytes + 127) / 128 * 128;
    const int fixed = 2 * g.b_bytes + 2 * kSWarps * 4 * kSMaxJ * kSMaxHalf * 4 + 2 * 16 * 4 + 256;
    g.Bo = 0;
    for (int bo = (p.OH < 8 ? p.OH : 8); bo >= 1; --bo) {
        const int Lv = (bo - 1) * g.E + g.OWt;
        const int Tn = (Lv + g.TS - 1) / g.TS;
        const int maxe = ((p.KH - 1) / 2) * g.E + (Tn - 1) * g.TS + 127;
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
    g.bias_off = g.x_off + 2 * kSWarps * 4 * kSMaxJ * kSMaxHalf * 4;
    g.bar_off = g.bias_off + 2 * 16 * 4;
    g.smem = g.bar_off + 256;
    if (g.smem > kSSmemCap) return false;
    int cols = kSTileBufs * g.N, pow2 = 32;
    while (pow2 < cols) pow2 *= 2;
    if (pow2 > 512) return false;
    g.tmem_cols = pow2;
    g.idesc = s_idesc(p.dtype == GCONV_BF16, 128, g.N);
    g.Ediv = FastDiv((uint32_t)g.E);
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

__device__ __forceinline__ bool s_wait(uint32_t bar, uint32_t parity, volatile int *failed) {
    for (uint32_t i = 0; i < kSSpinLimit; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
        if (*failed) return false;
    }
    *failed = 1;
    return false;
}
// The same wait, bounded but ignoring the failure flag (the clean-up path).
__device__ __forceinline__ void s_wait_final(uint32_t bar, uint32_t parity) {
    for (uint32_t i = 0; i < kSSpinLimit; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return;
    }
}
__device__ __forceinline__ void s_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void s_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void s_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void s_mma(uint32_t tmem, uint64_t adesc, uint64_t bdesc,
                                      uint32_t idesc, int accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void s_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
        : "memory");
}
template <int NC>
__device__ __forceinline__ void s_ld(uint32_t taddr, float (&v)[NC]);
template <>
__device__ __forceinline__ void s_ld<8>(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
template <>
__device__ __forceinline__ void s_ld<4>(uint32_t taddr, float (&v)[4]) {
    uint32_t r[4];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void s_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void s_producer_sync() {   // warps 0-7 only
    asm volatile("bar.sync 1, %0;\n" ::"n"(kSProducers) : "memory");
}

// T: element type; HALF: output channels per drain warp (NN / 2).
template <typename T, int HALF>
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

    // mbarriers: staged[2] (the unit's four boxes landed + weights and bias
    // written: 1 expect-tx arrival + 256 producer arrivals), ring_free[2]
    // (every MMA that read the unit buffer completed: one commit per
    // issuer), acc_full[4] (a tile's MMAs completed), acc_empty[4] (a tile
    // drained: 256 arrivals).
    const uint32_t bar_staged = sbase + (uint32_t)g.bar_off;
    const uint32_t bar_free = bar_staged + 16u;
    const uint32_t bar_full = bar_staged + 32u;
    const uint32_t bar_empty = bar_staged + 64u;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(s_smem + g.bar_off + 96);
    volatile int *failed = reinterpret_cast<volatile int *>(s_smem + g.bar_off + 100);
    float *bias_s = reinterpret_cast<float *>(s_smem + g.bias_off);   // [2][16]
    float *xch = reinterpret_cast<float *>(s_smem + g.x_off);        // [2][8 warps][4][J][HALF]

    if (warp == kSWarps) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                         sbase + (uint32_t)(g.bar_off + 96)),
                     "r"(g.tmem_cols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
    }
    if (t == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_staged + 8u * i, kSProducers + 1);
            mbar_init(bar_free + 8u * i, kSIssuers);
        }
        for (int i = 0; i < kSTileBufs; ++i) {
            mbar_init(bar_full + 8u * i, 1);
            mbar_init(bar_empty + 8u * i, kSProducers);
        }
        *failed = 0;
        fence_barrier_init();
        tma_prefetch_map(&xmap);
    }
    s_fence_before();
    __syncthreads();
    s_fence_after();
    const uint32_t tmem = *tslot;

    if (warp >= kSWarps) {
        // ---------------- MMA issue: issuer i takes tiles i, i+2, ... -------
        const int iss = warp - kSWarps;
        if (lane == 0) {
            const uint32_t lbo = (uint32_t)(2 * g.arr_bytes);   // ph = 1 array of the same s
            int gt = 0;
            for (int k = 0; k < nunits; ++k) {
                const int ub = k & 1;
                s_wait(bar_staged + 8u * ub, (uint32_t)((k >> 1) & 1), failed);
                s_fence_after();
                const uint32_t ring = sbase + (uint32_t)g.ring_off[ub];
                const uint32_t bb = sbase + (uint32_t)g.b_off[ub];
                for (int tt = 0; tt < g.Tn; ++tt, ++gt) {
                    if ((gt & 1) != iss) continue;
                    const int tb = gt & (kSTileBufs - 1);
                    const int use = gt / kSTileBufs;
                    if (use >= 1) s_wait(bar_empty + 8u * tb, (uint32_t)((use - 1) & 1), failed);
                    s_fence_after();
                    if (!*failed) {
                        const uint32_t d = tmem + (uint32_t)(tb * g.N);
                        for (int kh = 0; kh < p.KH; ++kh) {
                            const int s = kh & 1, kr = kh >> 1;
                            const uint32_t a = ring + (uint32_t)(s * g.arr_bytes) +
                                               (uint32_t)((kr * g.E + tt * g.TS) * 16);
                            const uint64_t ad = s_desc(a, lbo, 128);
                            const uint64_t bd = s_desc(bb + (uint32_t)(kh * g.N * 32), 128, 256);
                            s_mma(d, ad, bd, g.idesc, kh);
                        }
                    }
                    s_commit(bar_full + 8u * tb);
                }
                s_commit(bar_free + 8u * ub);
            }
        }
        __syncwarp();
    } else {
        // ------------- staging and tensor-memory drain (warps 0-7) -------------
        const uint32_t box_bytes = (uint32_t)(16 * g.E * g.R);
        // Chunk c's weights into buffer ub: slice kh is an N x 16 K-major
        // block, row n = j*NN + n' (output channel c*NN + n'), K = ph*8 + cc
        // (chunk channel cc); zero outside the kernel and n''s group.
        auto stage_b = [&](int c, int ub) {
            T *bsm = reinterpret_cast<T *>(s_smem + g.b_off[ub]);
            const int total = p.KH * g.N * 16;
            for (int e = t; e < total; e += kSProducers) {
                const int kk = e & 15;
                const int n = (e >> 4) % g.N;
                const int kh = (e >> 4) / g.N;
                const int j = n / g.NN, np = n - j * g.NN;
                const int ph = kk >> 3, cc = kk & 7;
                const int kw = 2 * j + ph - g.dc;
                const int cb = (np / p.Cout_g) * p.Cin_g;
                float v = 0.f;
                if (j < g.J && kw >= 0 && kw < p.KW && cc >= cb && cc < cb + p.Cin_g) {
                    const int co = c * g.NN + np;
                    v = load_f32(w + (int64_t)co * p.ws[0] + (int64_t)(cc - cb) * p.ws[1] +
                                 (int64_t)kh * p.ws[2] + (int64_t)kw * p.ws[3]);
                }
                const int off = kh * g.N * 32 + (n >> 3) * 256 + (kk >> 3) * 128 + (n & 7) * 16 +
                                (kk & 7) * 2;
                *reinterpret_cast<T *>(reinterpret_cast<unsigned char *>(bsm) + off) =
                    from_f32<T>(v);
            }
        };
        int b_chunk[2] = {-1, -1};
        // Stage unit u into buffer ub (k-th unit of this CTA): thread 0 waits
        // until the unit two back has been read by the tensor core, then
        // issues the four boxes; the weights are restaged when the chunk of
        // this buffer changes (after the same wait).  Every producer then
        // arrives on staged[ub].
        auto stage = [&](const TcsUnit &u, int k) {
            const int ub = k & 1;
            const bool new_b = b_chunk[ub] != u.c;
            // every producer has finished draining the unit that last used
            // this buffer's bias
            s_producer_sync();
            if (k >= 2 && (t == 0 || new_b))
                s_wait(bar_free + 8u * ub, (uint32_t)(((k - 2) >> 1) & 1), failed);
            if (t == 0) {
                mbar_arrive_expect_tx(bar_staged + 8u * ub, 4u * box_bytes);
                const int oh0 = u.b * g.Bo, ow0 = u.ct * g.OWt;
                const uint32_t ring = sbase + (uint32_t)g.ring_off[ub];
                for (int a = 0; a < 4; ++a) {
                    const int ph = a >> 1, s = a & 1;
                    tma_load_4d(ring + (uint32_t)((ph * 2 + s) * g.arr_bytes), &xmap,
                                bar_staged + 8u * ub, 8 * u.c, 2 * ow0 - g.cpad + ph,
                                2 * oh0 - p.pbh + s, u.n);
                }
            }
            if (new_b) {
                stage_b(u.c, ub);
                b_chunk[ub] = u.c;
            }
            if (t < g.NN)
                bias_s[ub * 16 + t] =
                    p.has_bias ? load_f32(b + (int64_t)(u.c * g.NN + t) * p.bs) : 0.f;
            asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
            s_arrive(bar_staged + 8u * ub);
        };

        // Drain tile tt of unit u (global tile gt): warp (qd, hf) reads its
        // 32 accumulator rows' HALF columns of every shift j, adds the
        // shifted rows (shuffles inside the warp, the next warp's first
        // rows through shared memory), the bias, rounds once, stores.
        const int qd = warp & 3, hf = warp >> 2;
        auto drain = [&](const TcsUnit &u, int k, int tt, int gt) {
            const int ub = k & 1;
            const int tb = gt & (kSTileBufs - 1);
            s_wait(bar_full + 8u * tb, (uint32_t)((gt / kSTileBufs) & 1), failed);
            s_fence_after();
            float a[kSMaxJ][HALF];
            const uint32_t taddr = tmem + ((uint32_t)(32 * qd) << 16) +
                                   (uint32_t)(tb * g.N + hf * HALF);
#pragma unroll
            for (int j = 0; j < kSMaxJ; ++j)
                if (j < g.J) s_ld<HALF>(taddr + (uint32_t)(j * g.NN), a[j]);
            s_wait_ld();
            s_fence_before();
            s_arrive(bar_empty + 8u * tb);
            // rows 0 .. J-2 of this warp, for the warp holding the rows below
            float *xw = xch + ((gt & 1) * kSWarps + warp) * (4 * kSMaxJ * kSMaxHalf);
            if (lane < g.J - 1) {
#pragma unroll
                for (int j = 1; j < kSMaxJ; ++j)
#pragma unroll
                    for (int c = 0; c < HALF; ++c)
                        if (j < g.J) xw[(lane * kSMaxJ + j) * kSMaxHalf + c] = a[j][c];
            }
            s_producer_sync();
            const float *xn = xch + ((gt & 1) * kSWarps + (warp + 1)) * (4 * kSMaxJ * kSMaxHalf);
            float acc[HALF];
#pragma unroll
            for (int c = 0; c < HALF; ++c) acc[c] = a[0][c];
#pragma unroll
            for (int j = 1; j < kSMaxJ; ++j) {
                if (j >= g.J) break;
#pragma unroll
                for (int c = 0; c < HALF; ++c) {
                    float v = __shfl_down_sync(0xffffffffu, a[j][c], j);
                    if (lane + j >= 32) v = qd < 3 ? xn[((lane + j - 32) * kSMaxJ + j) * kSMaxHalf + c] : 0.f;
                    acc[c] += v;
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
            const bool bad = *failed != 0;
            float f[HALF];
#pragma unroll
            for (int c = 0; c < HALF; ++c)
                f[c] = bad ? __int_as_float(0x7fc00000) : acc[c] + bias_s[ub * 16 + hf * HALF + c];
            const int co0 = u.c * g.NN + hf * HALF;
            T *yp = y + (int64_t)u.n * p.ys[0] + (int64_t)oh * p.ys[2] + (int64_t)ow * p.ys[3] +
                    (int64_t)co0 * p.ys[1];
            if (g.vec_store) {
                if constexpr (HALF == 8) {
                    uint4 o;
                    o.x = pack2(f[0], f[1], (T *)nullptr);
                    o.y = pack2(f[2], f[3], (T *)nullptr);
                    o.z = pack2(f[4], f[5], (T *)nullptr);
                    o.w = pack2(f[6], f[7], (T *)nullptr);
                    *reinterpret_cast<uint4 *>(yp) = o;
                } else {
                    uint2 o;
                    o.x = pack2(f[0], f[1], (T *)nullptr);
                    o.y = pack2(f[2], f[3], (T *)nullptr);
                    *reinterpret_cast<uint2 *>(yp) = o;
                }
            } else {
#pragma unroll
                for (int c = 0; c < HALF; ++c) yp[(int64_t)c * p.ys[1]] = from_f32<T>(f[c]);
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
            for (int tt = 0; tt < g.Tn; ++tt, ++gt) drain(cur, k, tt, gt);
            cur = nxt;
            nxt.next(g, p.N);
        }
    }
    // Clean-up: after a failed wait, wait (bounded) for the last unit's
    // boxes and MMAs before the shared and tensor memory go away.
    s_fence_before();
    __syncthreads();
    s_fence_after();
    if (t == 0) {
        // the last unit's commits (and, after a failure, its boxes) have
        // landed before the barriers' memory is released
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
    const uint32_t box[4] = {8u, (uint32_t)(2 * g.E), (uint32_t)(2 * g.R), 1u};
    const uint32_t estr[4] = {1u, 2u, 2u, 1u};
    if (!tma_encode_4d_strided(&map, tma_dtype<T>(), q.x, dims, strides, box, estr))
        return cudaErrorInvalidValue;
    cudaError_t e;
    if (g.NN == 16) {
        e = cudaFuncSetAttribute(tcs_kernel<T, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 g.smem);
        if (e != cudaSuccess) return e;
        e = launch_pdl(tcs_kernel<T, 8>, dim3(g.ctas), dim3(kSThreads), g.smem, s, map,
                       static_cast<const T *>(q.w), static_cast<const T *>(q.b),
                       static_cast<T *>(q.y), p, g);
    } else {
        e = cudaFuncSetAttribute(tcs_kernel<T, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 g.smem);
        if (e != cudaSuccess) return e;
        e = launch_pdl(tcs_kernel<T, 4>, dim3(g.ctas), dim3(kSThreads), g.smem, s, map,
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
    const int half = g.NN / 2;
    g.vec_store = aligned(q.y, 2 * half) && p.ys[1] == 1 && p.ys[3] % half == 0 &&
                  p.ys[2] % half == 0 && p.ys[0] % half == 0;
    if (p.dtype == GCONV_BF16) return tcs_launch_t<__nv_bfloat16>(p, q, s, g);
    return tcs_launch_t<__half>(p, q, s, g);
}

}  // namespace gconv
