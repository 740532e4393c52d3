// k_tc.cu -- grp_tc: few-channel grouped convolution (4 or 8 input channels
// per group, channels-last, bf16/fp16) as an implicit GEMM on the
// fifth-generation tensor cores: tcgen05.mma kind::f16 with fp32
// accumulators in tensor memory (TMEM).
//
// The convolution is the one of torch/_inductor/kernel/conv.py
// (LOOP_BODY_2D indexing, conv2d_template group offsets); executorch
// PR #25085 (description, second paragraph) leaves grouped convolutions
// whose per-group matrix product suits a tensor-core template to that
// template.  This schedule is that matrix product, written for sm_103a:
//
//  - An 8-channel chunk of the input (16 bytes per pixel) holds 8 / Cin_g
//    whole groups.  For one chunk the product is
//      Y[m][n] = sum over taps t and chunk channels c of A[m][t,c] B[n][t,c]
//    with m an output pixel, n one of the chunk's NN = (8 / Cin_g) * Cout_g
//    output channels and B zero where channel c is not in n's group.
//  - A tile is M = 64 output pixels of one output row.  The input rows the
//    tile reads are staged in shared memory as stride-phase arrays of
//    16-byte entries (entry j of phase p of staged row r = input pixel
//    (ih0 + r, iw0 + j*SW + p)), filled by cp.async with zero fill for the
//    padding.  For tap (kh, kw) the 64 rows of A are then 64 consecutive
//    entries, i.e. a K-major, unswizzled operand whose 8x16-byte core
//    matrices are contiguous: no im2col copy is made.  One MMA (K = 16)
//    takes two taps of the same phase; its second 8-element K slice sits
//    one entry further on (leading byte offset 16).
//  - B (the chunk's weights) is staged once per chunk in the canonical
//    K-major layout, its K slices in the order the MMAs consume them.
//  - A work unit is R output rows of one (image, ow tile, chunk); R
//    threads in separate warps each issue one row's taps / 2 MMAs into
//    that row's NN TMEM columns and commit them to one mbarrier.  Units are double-buffered:
//    while the tensor core works on unit k, the CTA stages unit k+1 and
//    drains unit k-1 from TMEM (tcgen05.ld), adds the bias in fp32, rounds
//    once and stores 16-byte vectors.  Two CTAs share an SM (eight MMA
//    issuers; an M = 64 MMA uses half of the tensor core's lanes).
//  - Every mbarrier wait is bounded; a wait that gives up marks the CTA
//    failed, its outputs are written as NaN and no TMEM is freed before the
//    MMAs it issued have been waited for once more.
#include <cstdint>

#include "device_common.cuh"
#include "gconv_internal.h"
#include "launch.cuh"
#include "tma.cuh"

namespace gconv {
namespace {

constexpr int kTcProducers = 128;   // warps 0-3: staging and TMEM drain
constexpr int kTcIssuers = 4;       // warps 4-7: MMA issue, one output row each
constexpr int kTcThreads = kTcProducers + 32 * kTcIssuers;
constexpr int kTcMT = 64;          // output pixels per tile (MMA M)
constexpr int kTcMaxMMA = 48;      // tap pairs per output row (9x9: 45)
constexpr int kTcSmemCap = 112 * 1024;   // two CTAs per SM
constexpr int kTcCtasPerSM = 2;

struct TcGeom {
    int gpc;        // groups per 8-channel chunk (8 / Cin_g)
    int NN;         // output channels per chunk (MMA N)
    int chunks;     // C_in / 8
    int R;          // output rows per unit
    int rows_in;    // staged input rows per unit
    int NJ;         // entries per staged phase row
    int owt, obk;   // ow tiles, output-row blocks
    int nmma;       // MMAs (tap pairs) per output row
    int tap[kTcMaxMMA];   // kh | phase << 4 | s0 << 8 | kw0 << 12 | kw1 << 16 (kw1 15: none)
    int a_off[2];   // shared-memory byte offsets
    int b_off, tab_off, bias_off, bar_off, smem;
    int stage_bytes, b_sbo;   // A stage bytes, B stride between 8-row groups
    int tmem_cols;
    int units, ctas;
    uint32_t idesc;
    int vec_store;
};

// 64-bit shared-memory matrix descriptor (tcgen05): K-major, no swizzle.
// Start address, leading byte offset (between the two K-adjacent 8x16-byte
// core matrices) and stride byte offset (between M/N-adjacent ones), all
// in 16-byte units; bits 46-48 hold the descriptor version (1).
__device__ __forceinline__ uint64_t tc_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo & 0x3FFFFu) >> 4) << 16) |
           ((uint64_t)((sbo & 0x3FFFFu) >> 4) << 32) | ((uint64_t)1 << 46);
}

// 32-bit instruction descriptor for kind::f16: fp32 accumulator (bits
// 4-5 = 1), A and B both bf16 (1) or both fp16 (0) at bits 7-9 / 10-12,
// both K-major, N / 8 at bits 17-22, M / 16 at bits 24-28.
inline uint32_t tc_idesc(bool bf16, int M, int N) {
    const uint32_t ab = bf16 ? 1u : 0u;
    return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

bool tc_geometry(const Params &p, TcGeom &g) {
    if (p.Cin_g != 4 && p.Cin_g != 8) return false;
    if (p.C_in % 8 != 0) return false;
    if (p.sw != 1 && p.sw != 2) return false;
    g.gpc = 8 / p.Cin_g;
    g.NN = g.gpc * p.Cout_g;
    if (g.NN % 8 != 0 || g.NN > 32) return false;
    g.chunks = p.C_in / 8;
    g.R = 4;
    if (p.OH < g.R) g.R = p.OH;
    g.rows_in = (g.R - 1) * p.sh + p.KH;
    const int smax = (p.KW - 1) / p.sw;
    g.NJ = kTcMT + smax + 2;
    g.owt = (p.OW + kTcMT - 1) / kTcMT;
    g.obk = (p.OH + g.R - 1) / g.R;
    g.nmma = 0;
    for (int kh = 0; kh < p.KH; ++kh)
        for (int ph = 0; ph < p.sw; ++ph)
            for (int kw = ph; kw < p.KW; kw += 2 * p.sw) {
                if (g.nmma >= kTcMaxMMA) return false;
                const int kw1 = kw + p.sw < p.KW ? kw + p.sw : 15;
                g.tap[g.nmma++] = kh | (ph << 4) | ((kw / p.sw) << 8) | (kw << 12) | (kw1 << 16);
            }
    g.stage_bytes = g.rows_in * p.sw * g.NJ * 16;
    g.b_sbo = 2 * g.nmma * 128;
    const int b_bytes = (g.NN / 8) * g.b_sbo;
    g.a_off[0] = 0;
    g.a_off[1] = (g.stage_bytes + 1023) / 1024 * 1024;
    g.b_off = g.a_off[1] + (g.stage_bytes + 1023) / 1024 * 1024;
    g.tab_off = g.b_off + (b_bytes + 127) / 128 * 128;
    g.bias_off = g.tab_off + 2 * 4 * kTcMaxMMA * 16;   // descriptor table [buf][rr][mma]
    g.bar_off = g.bias_off + 2 * 32 * 4;
    g.smem = g.bar_off + 64;   // six mbarriers, TMEM address slot, failure flag
    if (g.smem > kTcSmemCap) return false;
    int cols = 2 * g.R * g.NN, pow2 = 32;
    while (pow2 < cols) pow2 *= 2;
    if (pow2 > 512 / kTcCtasPerSM) return false;
    g.tmem_cols = pow2;
    const int64_t units = (int64_t)g.chunks * p.N * g.obk * g.owt;
    if (units > INT32_MAX) return false;
    g.units = (int)units;
    const int cap = 152 * kTcCtasPerSM;
    g.ctas = g.units < cap ? g.units : cap;
    g.idesc = tc_idesc(p.dtype == GCONV_BF16, kTcMT, g.NN);
    g.vec_store = 0;
    return true;
}

// Division-free cursor over units (ow tile fastest, then row block, image,
// chunk): consecutive units of a CTA share the chunk's weights.
struct TcUnit {
    int c, n, ob, ot;
    __device__ __forceinline__ void set(int u, const TcGeom &g, int N) {
        ot = u % g.owt;
        int r = u / g.owt;
        ob = r % g.obk;
        r /= g.obk;
        n = r % N;
        c = r / N;
    }
    __device__ __forceinline__ void next(const TcGeom &g, int N) {
        if (++ot < g.owt) return;
        ot = 0;
        if (++ob < g.obk) return;
        ob = 0;
        if (++n < N) return;
        n = 0;
        ++c;
    }
};

__device__ __forceinline__ void tc_alloc(uint32_t slot, int cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(slot),
                 "r"(cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
}
__device__ __forceinline__ void tc_dealloc(uint32_t tmem, int cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(cols));
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
// D[tmem] (+)= A * B^T for one M x N x 16 step; accumulate selects D += .
__device__ __forceinline__ void tc_mma(uint32_t tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, int accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
// Arrive on the mbarrier once every MMA this thread issued has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                     bar)
                 : "memory");
}
// Eight fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tc_ld8(uint32_t taddr, uint32_t (&v)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                   "=r"(v[6]), "=r"(v[7])
                 : "r"(taddr));
}
__device__ __forceinline__ void tc_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tc_cp16(uint32_t dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

// Bounded wait on an mbarrier phase.  Gives up (returns false) after
// kTcSpinLimit polls or as soon as the CTA is marked failed, so one lost
// arrival never turns into a chain of long waits.
constexpr uint32_t kTcSpinLimit = 1u << 22;
__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, volatile int *failed) {
    for (uint32_t i = 0; i < kTcSpinLimit; ++i) {
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
__device__ __forceinline__ void tc_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_producer_sync() {   // warps 0-3 only
    asm volatile("bar.sync 1, %0;\n" ::"n"(kTcProducers) : "memory");
}

template <typename T, int SW>
__global__ void __launch_bounds__(kTcThreads, kTcCtasPerSM)
tc_kernel(const T *__restrict__ x, const T *__restrict__ w, const T *__restrict__ b,
          T *__restrict__ y, Params p, TcGeom g) {
    // Let the next kernel in the stream start launching; wait for the
    // previous kernel's memory before reading global memory.
    pdl_launch_dependents();
    pdl_wait();
    extern __shared__ __align__(1024) unsigned char tc_smem[];
    const uint32_t sbase = smem_addr(tc_smem);
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int per = g.units / g.ctas, extra = g.units % g.ctas;
    const int u0 = blockIdx.x * per + min((int)blockIdx.x, extra);
    const int nunits = per + ((int)blockIdx.x < extra ? 1 : 0);
    if (nunits <= 0) return;   // the same for the whole CTA

    // Complete (A, B) descriptor pairs of every MMA of a unit, per buffer and
    // output row: [buf][rr][mma] as {A lo, A hi, B lo, B hi}.
    uint4 *dtab = reinterpret_cast<uint4 *>(tc_smem + g.tab_off);
    float *bias_s = reinterpret_cast<float *>(tc_smem + g.bias_off);   // [2][32]
    // mbarriers: full[2] (rows + weights staged, 128 arrivals), done[2]
    // (the unit's MMAs completed: one tcgen05.commit per issuer), empty[2]
    // (TMEM block drained, 128 arrivals).
    const uint32_t bar_full = sbase + (uint32_t)g.bar_off;
    const uint32_t bar_done = bar_full + 16u;
    const uint32_t bar_empty = bar_full + 32u;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(tc_smem + g.bar_off + 48);
    volatile int *failed = reinterpret_cast<volatile int *>(tc_smem + g.bar_off + 52);
    T *bsm = reinterpret_cast<T *>(tc_smem + g.b_off);

    if (warp == 4) tc_alloc(sbase + (uint32_t)(g.bar_off + 48), g.tmem_cols);
    if (t == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_full + 8u * i, kTcProducers);
            mbar_init(bar_done + 8u * i, kTcIssuers);
            mbar_init(bar_empty + 8u * i, kTcProducers);
        }
        *failed = 0;
        fence_barrier_init();
    }
    for (int idx = t; idx < 2 * 4 * kTcMaxMMA; idx += kTcThreads) {
        const int i = idx % kTcMaxMMA, rr = (idx / kTcMaxMMA) % 4, buf = idx / (4 * kTcMaxMMA);
        const int e = i < g.nmma ? g.tap[i] : g.tap[0];   // padded entries are never issued
        const int off = (rr * p.sh * SW + (e & 15) * SW + ((e >> 4) & 15)) * g.NJ + ((e >> 8) & 15);
        const uint64_t a = tc_desc(sbase + (uint32_t)g.a_off[buf] + (uint32_t)(16 * off), 16, 128);
        const uint64_t bd = tc_desc(sbase + (uint32_t)g.b_off + (uint32_t)(256 * i), 128,
                                    (uint32_t)g.b_sbo);
        dtab[idx] = make_uint4((uint32_t)a, (uint32_t)(a >> 32), (uint32_t)bd, (uint32_t)(bd >> 32));
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp >= 4) {
        // ------- MMA issue: lane 0 of warp 4 + rr issues output row rr -------
        // One thread issues a small MMA every ~30 ns at best, well below the
        // tensor core's rate for these shapes; four issuers per CTA (eight
        // per SM) bring the SM to ~12-14 ns per MMA.  An issuer without a
        // row (R < 4) still arrives on done, so every unit's phase completes.
        const int rr = warp - 4;
        if (lane == 0) {
            for (int k = 0; k < nunits; ++k) {
                const int buf = k & 1;
                tc_wait(bar_full + 8u * buf, (uint32_t)((k >> 1) & 1), failed);
                if (k >= 2) tc_wait(bar_empty + 8u * buf, (uint32_t)(((k - 2) >> 1) & 1), failed);
                tc_fence_after();
                if (rr >= g.R) {
                    tc_arrive(bar_done + 8u * buf);
                    continue;
                }
                {
                    const uint32_t d = tmem + (uint32_t)((buf * g.R + rr) * g.NN);
                    const uint4 *row = dtab + (buf * 4 + rr) * kTcMaxMMA;
                    for (int i0 = 0; i0 < g.nmma; i0 += 8) {
                        uint4 v[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) v[j] = row[i0 + j];
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            if (i0 + j < g.nmma)
                                tc_mma(d, ((uint64_t)v[j].y << 32) | v[j].x,
                                       ((uint64_t)v[j].w << 32) | v[j].z, g.idesc, i0 + j);
                    }
                }
                tc_commit(bar_done + 8u * buf);
            }
        }
        __syncwarp();
    } else {
        // ------------- staging and TMEM drain (warps 0-3) -------------
        auto stage_a = [&](const TcUnit &u, int buf) {
            const uint32_t dst0 = sbase + (uint32_t)g.a_off[buf];
            const int ih0 = u.ob * g.R * p.sh - p.pbh;
            const int iw0 = u.ot * kTcMT * SW - p.pbw;
            const T *xc = x + (int64_t)u.n * p.xs[0] + (int64_t)(8 * u.c) * p.xs[1];
            for (int rp = warp; rp < g.rows_in * SW; rp += kTcProducers / 32) {
                const int r = rp / SW, ph = rp - r * SW;
                const int ih = ih0 + r;
                const bool row_ok = ih >= 0 && ih < p.H;
                const T *xrow = xc + (int64_t)(row_ok ? ih : 0) * p.xs[2];
                for (int j = lane; j < g.NJ; j += 32) {
                    const int iw = iw0 + j * SW + ph;
                    const bool ok = row_ok && iw >= 0 && iw < p.W;
                    tc_cp16(dst0 + (uint32_t)((rp * g.NJ + j) * 16),
                            ok ? (const void *)(xrow + (int64_t)iw * p.xs[3]) : (const void *)x,
                            ok ? 16 : 0);
                }
            }
            asm volatile("cp.async.commit_group;\n" ::: "memory");
        };
        // Chunk c's weights: row n (output channel c*NN + n), K slice q =
        // 2*mma + half holds the 8 chunk channels of that tap as one
        // 16-byte vector; channels outside n's group (and a missing second
        // tap) are zero.  Each thread builds whole slices, QB at a time with
        // every load in flight before the stores.
        auto stage_b = [&](int c) {
            constexpr int QB = 4;
            const int nq = 2 * g.nmma;
            const int total = g.NN * nq;
            for (int e0 = t; e0 < total; e0 += QB * kTcProducers) {
                union { uint4 u; T e[8]; } v[QB];
                int dst[QB];
#pragma unroll
                for (int j = 0; j < QB; ++j) {
                    v[j].u = make_uint4(0u, 0u, 0u, 0u);
                    const int e = e0 + j * kTcProducers;
                    dst[j] = -1;
                    if (e < total) {
                        const int n = e / nq, q = e - n * nq;
                        const int tp = g.tap[q >> 1];
                        const int kh = tp & 15;
                        const int kw = (q & 1) ? ((tp >> 16) & 15) : ((tp >> 12) & 15);
                        const int co = c * g.NN + n;
                        const int cb = (n / p.Cout_g) * p.Cin_g;   // n's group's first chunk channel
                        if (kw < p.KW) {
                            const T *src = w + (int64_t)co * p.ws[0] + (int64_t)kh * p.ws[2] +
                                           (int64_t)kw * p.ws[3];
                            T vals[8];
#pragma unroll
                            for (int ci = 0; ci < 8; ++ci)
                                vals[ci] = ci < p.Cin_g ? src[(int64_t)ci * p.ws[1]] : from_f32<T>(0.f);
                            // the group sits at chunk channels cb .. cb + Cin_g - 1 (cb is 0 or 4)
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                v[j].e[i] = cb == 0 ? vals[i] : (i >= 4 ? vals[i - 4] : from_f32<T>(0.f));
                        }
                        dst[j] = ((n >> 3) * g.b_sbo + q * 128 + (n & 7) * 16) / 16;
                    }
                }
#pragma unroll
                for (int j = 0; j < QB; ++j)
                    if (dst[j] >= 0) reinterpret_cast<uint4 *>(bsm)[dst[j]] = v[j].u;
            }
        };
        // Stage unit u (buffer buf): its rows, and the chunk's weights when
        // the chunk changes; then make the writes visible to the tensor
        // core and arrive on full[buf].
        auto stage = [&](const TcUnit &u, int buf, bool new_chunk) {
            stage_a(u, buf);
            if (new_chunk) stage_b(u.c);
            if (t < g.NN)
                bias_s[buf * 32 + t] = p.has_bias ? load_f32(b + (int64_t)(u.c * g.NN + t) * p.bs) : 0.f;
            asm volatile("cp.async.wait_group 0;\n" ::: "memory");
            asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
            tc_arrive(bar_full + 8u * buf);
        };
        // Drain unit u from TMEM block buf: warp w holds tile rows
        // 16w..16w+15 in lanes 0-15 of its sub-partition (the M = 64
        // layout); add the bias in fp32, round once, store 16-byte vectors.
        auto epilogue = [&](const TcUnit &u, int buf) {
            const int ow = u.ot * kTcMT + 16 * warp + lane;
            const bool px_ok = lane < 16 && ow < p.OW;
            const int co0 = u.c * g.NN;
            const bool bad = *failed != 0;
            for (int rr = 0; rr < g.R; ++rr) {
                const int oh = u.ob * g.R + rr;
                if (oh >= p.OH) break;
                uint32_t v[4][8];
                const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16) +
                                       (uint32_t)((buf * g.R + rr) * g.NN);
#pragma unroll
                for (int nb = 0; nb < 4; ++nb)
                    if (nb * 8 < g.NN) tc_ld8(taddr + (uint32_t)(nb * 8), v[nb]);
                tc_wait_ld();
                if (!px_ok) continue;
                T *yp = y + (int64_t)u.n * p.ys[0] + (int64_t)oh * p.ys[2] +
                        (int64_t)ow * p.ys[3] + (int64_t)co0 * p.ys[1];
#pragma unroll
                for (int nb = 0; nb < 4; ++nb) {
                    if (nb * 8 >= g.NN) break;
                    float f[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        f[e] = __uint_as_float(v[nb][e]) + bias_s[buf * 32 + nb * 8 + e];
                    if (bad) {   // a failed CTA writes NaN
#pragma unroll
                        for (int e = 0; e < 8; ++e) f[e] = __int_as_float(0x7fc00000);
                    }
                    if (g.vec_store) {
                        uint4 o;
                        o.x = pack2(f[0], f[1], (T *)nullptr);
                        o.y = pack2(f[2], f[3], (T *)nullptr);
                        o.z = pack2(f[4], f[5], (T *)nullptr);
                        o.w = pack2(f[6], f[7], (T *)nullptr);
                        *reinterpret_cast<uint4 *>(yp + nb * 8) = o;
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            yp[(int64_t)(nb * 8 + e) * p.ys[1]] = from_f32<T>(f[e]);
                    }
                }
            }
        };

        TcUnit cur;
        cur.set(u0, g, p.N);
        TcUnit nxt = cur;
        nxt.next(g, p.N);
        stage(cur, 0, true);
        for (int k = 0; k < nunits; ++k) {
            const int buf = k & 1;
            // Every producer is done with unit k-1 (its bias slot and A
            // buffer are free to refill).
            tc_producer_sync();
            if (k + 1 < nunits) {
                const bool new_chunk = nxt.c != cur.c;
                // New weights may be written only once unit k's MMAs (the
                // last that read the old ones) have completed.
                if (new_chunk) tc_wait(bar_done + 8u * buf, (uint32_t)((k >> 1) & 1), failed);
                // A buffer buf^1 was last read by unit k-1's MMAs, whose
                // completion this thread saw before draining them.
                stage(nxt, buf ^ 1, new_chunk);
            }
            tc_wait(bar_done + 8u * buf, (uint32_t)((k >> 1) & 1), failed);
            tc_fence_after();
            epilogue(cur, buf);
            tc_fence_before();
            tc_arrive(bar_empty + 8u * buf);
            cur = nxt;
            nxt.next(g, p.N);
        }
    }
    // Every MMA has completed (each unit's completion was waited for above)
    // unless a wait gave up: then wait for the last unit's commit once more
    // before the tensor memory is released.
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 4) {
        if (*failed) {
            const int kl = nunits - 1;
            uint32_t done = 0;
            for (uint32_t i = 0; i < kTcSpinLimit && !done; ++i)
                asm volatile(
                    "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                    "selp.u32 %0, 1, 0, p;\n\t}"
                    : "=r"(done)
                    : "r"(bar_done + 8u * (uint32_t)(kl & 1)), "r"((uint32_t)((kl >> 1) & 1))
                    : "memory");
        }
        tc_dealloc(tmem, g.tmem_cols);
    }
}

bool tc_supports(const gconv_desc &d, const Ptrs &q) {
    if (!plain_forward(d)) return false;                    // dilation 1, forward
    if (tcs_supports(d, q)) return true;                    // the shift form
    if (d.layout != GCONV_LAYOUT_NHWC) return false;
    if (d.dtype != GCONV_BF16 && d.dtype != GCONV_F16) return false;   // kind::f16 operands
    if (d.KH > 9 || d.KW > 9) return false;
    // 16-byte cp.async of 8 channels: aligned base, channel stride 1,
    // pixel / row / image strides in whole 8-channel units.
    if (!aligned(q.x, 16)) return false;
    if (d.x_strides[1] != 1 || d.x_strides[3] % 8 || d.x_strides[2] % 8 || d.x_strides[0] % 8)
        return false;
    Params p = make_params(d);
    TcGeom g;
    return tc_geometry(p, g);
}

// Shared memory reserved per CTA: at least a third of the SM's, so no more
// than two CTAs share an SM and their TMEM blocks always fit at once (an
// allocation never waits for another CTA).
constexpr int kTcSmemFloor = 80 * 1024;

template <typename T, int SW>
cudaError_t tc_launch_t(const Params &p, const Ptrs &q, cudaStream_t s, const TcGeom &g) {
    const int smem = g.smem > kTcSmemFloor ? g.smem : kTcSmemFloor;
    cudaError_t e = cudaFuncSetAttribute(tc_kernel<T, SW>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = launch_kernel(tc_kernel<T, SW>, dim3(g.ctas), dim3(kTcThreads), smem, s,
                   static_cast<const T *>(q.x), static_cast<const T *>(q.w),
                   static_cast<const T *>(q.b), static_cast<T *>(q.y), p, g);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t tc_launch(const Params &p, const Ptrs &q, cudaStream_t s, int *launches) {
    if (tcs_takes(p, q.x)) return tcs_launch(p, q, s, launches);
    *launches = 1;
    TcGeom g;
    if (!tc_geometry(p, g)) return cudaErrorNotSupported;
    // 16-byte stores of 8 output channels
    g.vec_store = aligned(q.y, 16) && p.ys[1] == 1 && p.ys[3] % 8 == 0 && p.ys[2] % 8 == 0 &&
                  p.ys[0] % 8 == 0;
    if (p.dtype == GCONV_BF16)
        return p.sw == 1 ? tc_launch_t<__nv_bfloat16, 1>(p, q, s, g)
                         : tc_launch_t<__nv_bfloat16, 2>(p, q, s, g);
    return p.sw == 1 ? tc_launch_t<__half, 1>(p, q, s, g) : tc_launch_t<__half, 2>(p, q, s, g);
}

}  // namespace

const Schedule kGrpTc = {"grp_tc", tc_supports, tc_launch};

}  // namespace gconv
