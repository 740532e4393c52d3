// k_dwtcl.cu -- dw_tcl: channels-last depthwise convolution of bf16/fp16
// tensors at stride 1 on the tcgen05 tensor cores, the kernel's columns as a
// banded matrix, the input transposed to channel planes in shared memory.
//
// The operation is the depthwise case of the direct stencil of executorch
// PR #25085 (description, second paragraph; the channels-last layout is the
// one its schedules name for contiguous channels): y[n, oh, ow, c] =
// sum_{kh, kw} w[c, 0, kh, kw] * x[n, oh - pad_h + kh, ow - pad_w + kw, c].
// This form of it is written for sm_103a.  For one channel c, one kernel
// row kh and a tile of OWC = 17 - KW output columns starting at ow0:
//   D[r][j] += sum_k A[r + kh][k] * B[j][k],   k = 0 .. 15
// with A[rho][k] = x[., rho-th staged row, ow0 - pad_w + k, c] (M = 128
// output rows, K = 16 input columns) and the banded B[j][k] = w[c, kh, k - j]
// for j < OWC (zero outside the kernel, and for the rows j >= OWC).  Summed
// over kh in tensor memory, D[r][j] is the output at the row r maps to and
// column ow0 + j: the drain only adds the bias and rounds.
//  - Rows: a segment is a run of up to 128 output rows of one image (its
//    rows plus KH - 1 halo rows are staged); S segments whose staged rows
//    fit in 128 + KH - 1 are stacked along M (two 56-row images at once for
//    a 7x7 kernel), so short images still fill the 128-row MMA.  Output row
//    j of segment i is D row i * P + j (P = staged rows per segment); the D
//    rows between segments mix images and are not stored.
//  - A unit is one channel group of 8 channels, one stack of segments and
//    one column tile.  Its input (8 channels x 16 columns x P rows per
//    segment) is copied into a ring slot as 16-byte pieces, one per pixel,
//    by asynchronous copies from three warps (cp.async with a zero source
//    size for the padding), which an mbarrier tracks.  A 16-byte piece
//    every 2 C bytes is where the copy engine is slow (a box of such pieces
//    ran at about 0.16 pieces per cycle per SM); the load/store path takes
//    them at the rate of its cache-line requests, and one warp alone could
//    not issue them fast enough.  CTA i keeps channel group i mod (C / 8):
//    the groups' pieces of one pixel reach L2 at about the same time, from
//    sibling CTAs working through the same spatial units.
//    Two transposing warps turn each staged row
//    into the MMA operand: an ldmatrix of 8 pixels x 8 channels and a
//    transposing stmatrix give each channel's 8 consecutive columns as one
//    16-byte row of its K-major, unswizzled A (two 8-column chunks, a
//    chunk pitch apart; the channel planes an odd number of 16-byte units
//    apart, so the 8 rows of one stmatrix fall in different banks).  The
//    same warps build the group's banded weight matrices when the channel
//    group changes.
//  - Two warps issue the MMAs, four channels each (KH MMAs of N = 16 per
//    channel into tensor-memory columns 16 c of the unit's buffer); eight
//    warps drain tensor memory (two warpgroups taking alternate units),
//    three warps copy the input.  Tensor memory holds four unit buffers.
//  - Every mbarrier wait is bounded; a wait that gives up marks the CTA
//    failed, its outputs are written as NaN, and before exiting the CTA
//    waits (bounded) for its copies and MMAs in flight before it frees its
//    tensor memory.
#include <cstdint>

#include "device_common.cuh"
#include "gconv_internal.h"
#include "launch.cuh"
#include "tc_common.cuh"
#include "tma.cuh"   // smem_addr, mbarrier helpers

namespace gconv {
namespace {

using namespace tc;

constexpr int kLDrainWarps = 8;                   // tensor-memory drain
constexpr int kLTrans = 2;                        // transposing warps
constexpr int kLIssuers = 2;                      // MMA issue warps, 4 channels each
constexpr int kLLoaders = 3;                      // warps that copy the input
constexpr int kLWTrans = kLDrainWarps;            // first transposing warp
constexpr int kLWIssue = kLWTrans + kLTrans;      // first issuing warp
constexpr int kLWLoad = kLWIssue + kLIssuers;     // first copying warp
constexpr int kLThreads = 32 * (kLWLoad + kLLoaders);
constexpr int kLTransThreads = 32 * kLTrans;
constexpr int kLTmemBufs = 4;                     // unit buffers of 128 columns
constexpr int kLMaxSlots = 3;                     // input ring slots
constexpr int kLMaxABufs = 3;                     // A operand buffers
constexpr int kLSmemCap = 227 * 1024;

struct TclGeom {
    int Lo;            // output rows per segment
    int P;             // staged rows per segment: Lo + KH - 1
    int S;             // segments stacked along M
    int rbs;           // segments (row blocks) per image
    int nseg;          // segments in all
    int sgs;           // stacks of S segments
    int owc;           // output columns per tile: 17 - KW
    int cts;           // column tiles
    int cgs;           // channel groups of 8
    int RA;            // A rows: 128 + KH - 1
    int CH;            // A chunk pitch (RA rows of 16 bytes)
    int CP;            // A channel pitch: an odd number of 16-byte units >= 2 CH
    int slot_bytes;    // S * P staged rows of 16 columns x 8 channels
    int a_bytes, b_bytes;
    int NS, NA;        // ring slots, A buffers
    int a_off, b_off, bar_off, smem;
    int units, ctas;
    int wpc;           // CTAs per channel group (0: one contiguous split of all units)
    uint32_t idesc;
    int vec_store;     // 16-byte stores of 8 channels
};

bool tcl_geometry(const Params &p, TclGeom &g) {
    if (p.transposed || p.sh != 1 || p.sw != 1 || p.dh != 1 || p.dw != 1) return false;
    if (p.Cin_g != 1 || p.Cout_g != 1) return false;
    if (p.dtype != GCONV_BF16 && p.dtype != GCONV_F16) return false;
    if (p.KH < 1 || p.KH > 9 || p.KW < 1 || p.KW > 9) return false;
    if (p.C_in % 8 != 0 || p.OH < 1 || p.OW < 1) return false;
    g.Lo = p.OH < 128 ? p.OH : 128;
    g.P = g.Lo + p.KH - 1;
    g.S = (128 - g.Lo) / g.P + 1;
    g.rbs = (p.OH + g.Lo - 1) / g.Lo;
    const int64_t nseg = (int64_t)p.N * g.rbs;
    if (nseg > INT32_MAX / 2) return false;
    g.nseg = (int)nseg;
    g.sgs = (g.nseg + g.S - 1) / g.S;
    g.owc = 17 - p.KW;
    g.cts = (p.OW + g.owc - 1) / g.owc;
    g.cgs = p.C_in / 8;
    g.RA = 128 + p.KH - 1;
    g.CH = g.RA * 16;
    g.CP = 2 * g.CH;
    if (((g.CP >> 4) & 1) == 0) g.CP += 16;
    g.slot_bytes = g.S * g.P * 256;
    g.a_bytes = (8 * g.CP + 127) / 128 * 128;
    g.b_bytes = 8 * p.KH * 512;
    const int bars = 8 * (2 * kLMaxSlots + 2 * kLMaxABufs + 2 * kLTmemBufs + 1) + 16;
    // the deepest ring, then the most A buffers, that fit
    g.NS = 0;
    for (int ns = kLMaxSlots; ns >= 2 && !g.NS; --ns)
        for (int na = kLMaxABufs; na >= 2; --na)
            if (ns * g.slot_bytes + na * g.a_bytes + g.b_bytes + bars <= kLSmemCap) {
                g.NS = ns;
                g.NA = na;
                break;
            }
    if (!g.NS) return false;
    g.a_off = g.NS * g.slot_bytes;
    g.b_off = g.a_off + g.NA * g.a_bytes;
    g.bar_off = g.b_off + g.b_bytes;
    g.smem = g.bar_off + bars;
    // more than half an SM's shared memory: one CTA per SM, so a CTA never
    // waits for another's tensor memory
    if (g.smem < 120 * 1024) g.smem = 120 * 1024;
    const int64_t units = (int64_t)g.cgs * g.sgs * g.cts;
    if (units > INT32_MAX) return false;
    g.units = (int)units;
    // CTA i takes channel group i % cgs and the i / cgs-th share of the
    // spatial units, the same share as its sibling CTAs of the other groups:
    // the groups' 16-byte pieces of one pixel go through L2 at about the same
    // time (one DRAM fetch per line instead of one per piece) and a CTA
    // keeps one group's weights
    const int nsp = g.sgs * g.cts;
    g.wpc = g.cgs <= 152 ? 152 / g.cgs : 0;
    if (g.wpc > nsp) g.wpc = nsp;
    g.ctas = g.wpc ? g.wpc * g.cgs : 152;
    g.idesc = s_idesc(p.dtype == GCONV_BF16, 128, 16);
    g.vec_store = 0;
    return true;
}

// Division-free cursor over units (column tile fastest, then segment stack,
// then channel group).
struct TclUnit {
    int ct, sg, cg;
    __device__ __forceinline__ void set(int u, const TclGeom &g) {
        ct = u % g.cts;
        const int r = u / g.cts;
        sg = r % g.sgs;
        cg = r / g.sgs;
    }
    __device__ __forceinline__ void next(const TclGeom &g) {
        if (++ct < g.cts) return;
        ct = 0;
        if (++sg < g.sgs) return;
        sg = 0;
        ++cg;
    }
};

__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

template <typename T>
__global__ void __launch_bounds__(kLThreads, 1)
dwtcl_kernel(const T *__restrict__ x, const T *__restrict__ w,
             const T *__restrict__ b, T *__restrict__ y, Params p, TclGeom g) {
    pdl_launch_dependents();
    pdl_wait();
    extern __shared__ __align__(1024) unsigned char l_smem[];
    const uint32_t sbase = smem_addr(l_smem);
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    int u0, nunits;
    if (g.wpc) {   // one channel group, a contiguous share of its spatial units
        const int nsp = g.sgs * g.cts, cg = blockIdx.x % g.cgs, wk = blockIdx.x / g.cgs;
        const int per = nsp / g.wpc, extra = nsp % g.wpc;
        u0 = cg * nsp + wk * per + min(wk, extra);
        nunits = per + (wk < extra ? 1 : 0);
    } else {       // a contiguous share of all units
        const int per = g.units / g.ctas, extra = g.units % g.ctas;
        u0 = blockIdx.x * per + min((int)blockIdx.x, extra);
        nunits = per + ((int)blockIdx.x < extra ? 1 : 0);
    }
    if (nunits <= 0) return;

    // mbarriers: sfull[NS] (a slot's copies landed: one arrival per copying
    // thread), sfree[NS] (the slot is
    // transposed: 64 arrivals), aready[NA] (an A buffer written: 64),
    // afree[NA] (every MMA that read the A buffer completed: one commit per
    // issuer), full[4] (a unit's MMAs completed), empty[4] (a unit drained:
    // 128 arrivals), bready (the channel group's weights written: 64).  Unit
    // k uses slot k % NS, A buffer k % NA and tensor-memory buffer k % 4.
    const uint32_t bar_sfull = sbase + (uint32_t)g.bar_off;
    const uint32_t bar_sfree = bar_sfull + 8u * kLMaxSlots;
    const uint32_t bar_aready = bar_sfree + 8u * kLMaxSlots;
    const uint32_t bar_afree = bar_aready + 8u * kLMaxABufs;
    const uint32_t bar_full = bar_afree + 8u * kLMaxABufs;
    const uint32_t bar_empty = bar_full + 8u * kLTmemBufs;
    const uint32_t bar_bready = bar_empty + 8u * kLTmemBufs;
    const int slot_off = g.bar_off + 8 * (2 * kLMaxSlots + 2 * kLMaxABufs + 2 * kLTmemBufs + 1);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(l_smem + slot_off);
    volatile int *failed = reinterpret_cast<volatile int *>(l_smem + slot_off + 4);

    if (warp == kLWIssue) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                         sbase + (uint32_t)slot_off),
                     "r"(kLTmemBufs * 128));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
    }
    if (t == 0) {
        for (int i = 0; i < g.NS; ++i) {
            mbar_init(bar_sfull + 8u * i, 32 * kLLoaders);
            mbar_init(bar_sfree + 8u * i, kLTransThreads);
        }
        for (int i = 0; i < g.NA; ++i) {
            mbar_init(bar_aready + 8u * i, kLTransThreads);
            mbar_init(bar_afree + 8u * i, kLIssuers);
        }
        for (int i = 0; i < kLTmemBufs; ++i) {
            mbar_init(bar_full + 8u * i, kLIssuers);
            mbar_init(bar_empty + 8u * i, 128);
        }
        mbar_init(bar_bready, kLTransThreads);
        *failed = 0;
        fence_barrier_init();
    }
    s_fence_before();
    __syncthreads();
    s_fence_after();
    const uint32_t tmem = *tslot;

    if (warp >= kLWLoad) {
        // ------ input copies: unit k into slot k % NS once the slot's
        // previous unit is transposed.  Thread l of the copying warps copies
        // column l & 15 of every (2 kLLoaders)-th staged row from row l >> 4;
        // piece (row rho, column cc) of the slot sits at 16 (16 rho + cc)
        // bytes.  Each thread's arrival on the slot's mbarrier fires when its
        // own copies have landed. ------
        const int lt = t - 32 * kLWLoad;
        const int cc = lt & 15;
        TclUnit u;
        u.set(u0, g);
        for (int k = 0; k < nunits; ++k, u.next(g)) {
            const int sl = k % g.NS;
            if (k >= g.NS) s_wait_warp(bar_sfree + 8u * sl, (uint32_t)((k / g.NS - 1) & 1), failed);
            const int sa = min(g.S, g.nseg - u.sg * g.S);   // segments in this stack
            const uint32_t dst = sbase + (uint32_t)(sl * g.slot_bytes);
            const int iw = u.ct * g.owc - p.pbw + cc;
            const bool col_ok = iw >= 0 && iw < p.W;
            for (int i = 0; i < sa; ++i) {
                const int seg = u.sg * g.S + i;
                const int n = seg / g.rbs, rb = seg - n * g.rbs;
                const int row0 = rb * g.Lo - p.pbh;
                const T *xs = x + (int64_t)n * p.xs[0] + (int64_t)(col_ok ? iw : 0) * p.xs[3] + 8 * u.cg;
                for (int jr = lt >> 4; jr < g.P; jr += 2 * kLLoaders) {
                    const int ih = row0 + jr;
                    const bool ok = col_ok && ih >= 0 && ih < p.H;
                    const T *src = ok ? xs + (int64_t)ih * p.xs[2] : x;
                    const uint32_t sd = dst + (uint32_t)(((i * g.P + jr) * 16 + cc) * 16);
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(sd), "l"(src),
                                 "r"(ok ? 16 : 0)
                                 : "memory");
                }
            }
            asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar_sfull + 8u * sl)
                         : "memory");
        }
        // every copy of this thread has landed before the CTA can exit
        asm volatile("cp.async.wait_all;\n" ::: "memory");
    } else if (warp >= kLWIssue) {   // (warps kLWIssue .. kLWLoad - 1)
        // ------ MMA issue: issuer i takes channels 4i .. 4i + 3 of every unit ------
        const int iss = warp - kLWIssue;
        TclUnit u;
        u.set(u0, g);
        int prev_cg = -1, bstaged = 0;
        const uint64_t bd0 = s_desc(sbase + (uint32_t)g.b_off, 128, 256);
        for (int k = 0; k < nunits; ++k, u.next(g)) {
            const int ab = k % g.NA, tb = k % kLTmemBufs;
            if (u.cg != prev_cg) {   // the group's weights are rewritten
                prev_cg = u.cg;
                s_wait_warp(bar_bready, (uint32_t)(bstaged & 1), failed);
                ++bstaged;
            }
            s_wait_warp(bar_aready + 8u * ab, (uint32_t)((k / g.NA) & 1), failed);
            if (k >= kLTmemBufs)
                s_wait_warp(bar_empty + 8u * tb, (uint32_t)((k / kLTmemBufs - 1) & 1), failed);
            s_fence_after();
            if (!__any_sync(0xffffffffu, *failed != 0)) {
                // A of channel c starts at plane c, row kh (16 bytes a row);
                // the descriptors' start fields (16-byte units, no carry below
                // 2^18 bytes) advance by the offsets
                const uint64_t ad0 =
                    s_desc(sbase + (uint32_t)(g.a_off + ab * g.a_bytes), (uint32_t)g.CH, 128);
                // kernel row outer, channel inner: consecutive MMAs write
                // different accumulators, so none waits for the one before
#pragma unroll
                for (int kh = 0; kh < 9; ++kh) {
                    if (kh >= p.KH) break;
#pragma unroll
                    for (int cc = 0; cc < 8 / kLIssuers; ++cc) {
                        const int c = (8 / kLIssuers) * iss + cc;
                        s_mma_lane0(tmem + (uint32_t)(tb * 128 + c * 16),
                                    ad0 + (uint64_t)((c * g.CP + kh * 16) >> 4),
                                    bd0 + (uint64_t)(((c * p.KH + kh) * 512) >> 4), g.idesc, kh != 0,
                                    (uint32_t)lane);
                    }
                }
            }
            s_commit_lane0(bar_full + 8u * tb, (uint32_t)lane);
            s_commit_lane0(bar_afree + 8u * ab, (uint32_t)lane);
        }
    } else if (warp >= kLWTrans) {
        // ------ transposition of the staged rows and the weight matrices ------
        const int tw = warp - kLWTrans, tt = t - 32 * kLWTrans;
        // Channel group cg's banded matrices: block (c, kh) is a 16 x 16
        // K-major matrix whose row j holds at K = k the weight at kernel
        // column k - j (zero outside the kernel and for rows j >= OWC).  A
        // thread builds whole blocks: its KW weights load at once (the loads
        // overlap), and each row is the previous one shifted by a column.
        auto stage_b = [&](int cg) {
            unsigned char *bsm = l_smem + g.b_off;
            for (int blk = tt; blk < 8 * p.KH; blk += kLTransThreads) {
                const int c = blk / p.KH, kh = blk - c * p.KH;
                const T *wr = w + (int64_t)(8 * cg + c) * p.ws[0] + (int64_t)kh * p.ws[2];
                float row[16];
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    row[k] = (k < 9 && k < p.KW) ? load_f32(wr + (int64_t)k * p.ws[3]) : 0.f;
                unsigned char *dst = bsm + blk * 512;
#pragma unroll 1
                for (int j = 0; j < 16; ++j) {
                    const float on = j < g.owc ? 1.f : 0.f;
                    uint4 o[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        o[h].x = pack2(on * row[8 * h + 0], on * row[8 * h + 1], (T *)nullptr);
                        o[h].y = pack2(on * row[8 * h + 2], on * row[8 * h + 3], (T *)nullptr);
                        o[h].z = pack2(on * row[8 * h + 4], on * row[8 * h + 5], (T *)nullptr);
                        o[h].w = pack2(on * row[8 * h + 6], on * row[8 * h + 7], (T *)nullptr);
                    }
                    *reinterpret_cast<uint4 *>(dst + (j >> 3) * 256 + (j & 7) * 16) = o[0];
                    *reinterpret_cast<uint4 *>(dst + (j >> 3) * 256 + (j & 7) * 16 + 128) = o[1];
#pragma unroll
                    for (int k = 15; k > 0; --k) row[k] = row[k - 1];
                    row[0] = 0.f;
                }
            }
        };
        // ldmatrix lane roles: lane l gives row l & 7 of matrix l >> 3;
        // matrix m is staged row rho + (m >> 1), columns 8 (m & 1) .. + 7.
        const int mr = lane & 7, mq = (lane >> 3) & 1, md = lane >> 4;
        TclUnit u;
        u.set(u0, g);
        int prev_cg = -1;
        for (int k = 0; k < nunits; ++k, u.next(g)) {
            const int sl = k % g.NS, ab = k % g.NA;
            if (u.cg != prev_cg) {
                prev_cg = u.cg;
                // every MMA that read the previous group's weights has completed
                if (k >= 1)
                    s_wait_warp(bar_afree + 8u * (uint32_t)((k - 1) % g.NA),
                                (uint32_t)(((k - 1) / g.NA) & 1), failed);
                stage_b(u.cg);
                fence_async_smem();
                s_arrive(bar_bready);
            }
            s_wait_warp(bar_sfull + 8u * sl, (uint32_t)((k / g.NS) & 1), failed);
            if (k >= g.NA) s_wait_warp(bar_afree + 8u * ab, (uint32_t)((k / g.NA - 1) & 1), failed);
            const int rows = min(g.S, g.nseg - u.sg * g.S) * g.P;   // staged rows
            const uint32_t src = sbase + (uint32_t)(sl * g.slot_bytes);
            const uint32_t dst = sbase + (uint32_t)(g.a_off + ab * g.a_bytes);
            // pairs of staged rows, two pairs at a time (both loads in flight
            // before the stores); an odd last row, or a second pair past the
            // end, repeats the last row (same data to the same place)
            for (int rp = 4 * tw; rp < rows; rp += 4 * kLTrans) {
                const int rho0 = min(rp + md, rows - 1);
                const int rho1 = min(rp + 2 + md, rows - 1);
                const uint32_t la0 = src + (uint32_t)(rho0 * 256 + (8 * mq + mr) * 16);
                const uint32_t la1 = src + (uint32_t)(rho1 * 256 + (8 * mq + mr) * 16);
                uint32_t r[8];
                asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                             : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                             : "r"(la0));
                asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                             : "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                             : "r"(la1));
                // row mr of the transposed matrix is channel mr
                const uint32_t sa0 = dst + (uint32_t)(mr * g.CP + mq * g.CH + rho0 * 16);
                const uint32_t sa1 = dst + (uint32_t)(mr * g.CP + mq * g.CH + rho1 * 16);
                asm volatile(
                    "stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};\n" ::"r"(sa0),
                    "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
                    : "memory");
                asm volatile(
                    "stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};\n" ::"r"(sa1),
                    "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                    : "memory");
            }
            fence_async_smem();
            s_arrive(bar_aready + 8u * ab);
            s_arrive(bar_sfree + 8u * sl);
        }
    } else {
        // ------------- tensor-memory drain (warps 0-7) -------------
        // Warpgroup k & 1 drains unit k.  Thread r of the warpgroup holds D
        // row r: segment r / P, output row r % P of it.  It reads 8 columns
        // of the 8 channels at once, frees the buffer after the last read,
        // adds the bias, rounds once and stores 16 bytes (8 channels) per
        // output pixel.
        const int qd = warp & 3, wg = warp >> 2;
        const int r = 32 * qd + lane;
        const int si = r / g.P, sj = r - si * g.P;
        const uint32_t tlane = tmem + ((uint32_t)(32 * qd) << 16);
        TclUnit u;
        u.set(u0, g);
        for (int k = 0; k < nunits; ++k, u.next(g)) {
            if ((k & 1) != wg) continue;
            const int tb = k % kLTmemBufs;
            float bv[8];   // the bias loads go out before the wait
#pragma unroll
            for (int c = 0; c < 8; ++c)
                bv[c] = p.has_bias ? load_f32(b + (int64_t)(8 * u.cg + c) * p.bs) : 0.f;
            const int seg = u.sg * g.S + si;
            bool row_ok = si < g.S && sj < g.Lo && seg < g.nseg;
            int n = 0, oh = 0;
            if (row_ok) {
                n = seg / g.rbs;
                oh = (seg - n * g.rbs) * g.Lo + sj;
                row_ok = oh < p.OH;
            }
            const int ow0 = u.ct * g.owc;
            s_wait_warp(bar_full + 8u * tb, (uint32_t)((k / kLTmemBufs) & 1), failed);
            s_fence_after();
            const bool bad = *failed != 0;   // poison through the bias: NaN outputs
#pragma unroll
            for (int c = 0; c < 8; ++c)
                if (bad) bv[c] = __int_as_float(0x7fc00000);
            T *yrow = y + (int64_t)n * p.ys[0] + (int64_t)oh * p.ys[2] + (int64_t)(8 * u.cg) * p.ys[1];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (8 * h >= g.owc) break;
                float v[8][8];
                __syncwarp();
#pragma unroll
                for (int c = 0; c < 8; ++c)   // the whole warp
                    s_ld<8>(tlane + (uint32_t)(tb * 128 + c * 16 + 8 * h), v[c]);
                s_wait_ld();
                if (8 * h + 8 >= g.owc) {   // the buffer is read: free it
                    s_fence_before();
                    s_arrive(bar_empty + 8u * tb);
                }
                if (!row_ok) continue;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int col = 8 * h + e;
                    if (col >= g.owc || ow0 + col >= p.OW) break;
                    T *yp = yrow + (int64_t)(ow0 + col) * p.ys[3];
                    if (g.vec_store) {
                        uint4 o;
                        o.x = pack2(v[0][e] + bv[0], v[1][e] + bv[1], (T *)nullptr);
                        o.y = pack2(v[2][e] + bv[2], v[3][e] + bv[3], (T *)nullptr);
                        o.z = pack2(v[4][e] + bv[4], v[5][e] + bv[5], (T *)nullptr);
                        o.w = pack2(v[6][e] + bv[6], v[7][e] + bv[7], (T *)nullptr);
                        *reinterpret_cast<uint4 *>(yp) = o;
                    } else {
#pragma unroll
                        for (int c = 0; c < 8; ++c) yp[(int64_t)c * p.ys[1]] = from_f32<T>(v[c][e] + bv[c]);
                    }
                }
            }
        }
    }
    // Clean-up: the last unit's commits land before the shared and tensor
    // memory go away (the loader lanes waited for their own copies).
    s_fence_before();
    __syncthreads();
    s_fence_after();
    if (t == 0) {
        const int kl = nunits - 1;
        s_wait_final(bar_afree + 8u * (uint32_t)(kl % g.NA), (uint32_t)((kl / g.NA) & 1));
    }
    __syncthreads();
    if (warp == kLWIssue)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem),
                     "r"(kLTmemBufs * 128));
}

template <typename T>
cudaError_t dwtcl_launch_t(const Params &p, const Ptrs &q, cudaStream_t s, const TclGeom &g) {
    cudaError_t e =
        cudaFuncSetAttribute(dwtcl_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem);
    if (e != cudaSuccess) return e;
    e = launch_kernel(dwtcl_kernel<T>, dim3(g.ctas), dim3(kLThreads), g.smem, s,
                      static_cast<const T *>(q.x), static_cast<const T *>(q.w), static_cast<const T *>(q.b),
                      static_cast<T *>(q.y), p, g);
    return e != cudaSuccess ? e : cudaGetLastError();
}

bool dwtcl_takes(const Params &p, const void *x) {
    // 16-byte copies of 8 channels: 16-byte aligned base, channel stride 1,
    // column / row / image strides in whole 16-byte units.
    if (!aligned(x, 16)) return false;
    if (p.xs[1] != 1 || p.xs[3] % 8 || p.xs[2] % 8 || p.xs[0] % 8) return false;
    TclGeom g;
    return tcl_geometry(p, g);
}

bool dwtcl_supports(const gconv_desc &d, const Ptrs &q) {
    return !d.transposed && dwtcl_takes(make_params(d), q.x);
}

cudaError_t dwtcl_launch(const Params &p, const Ptrs &q, cudaStream_t s, int *launches) {
    *launches = 1;
    TclGeom g;
    if (!tcl_geometry(p, g)) return cudaErrorNotSupported;
    // 16-byte stores of 8 channels
    g.vec_store = aligned(q.y, 16) && p.ys[1] == 1 && p.ys[3] % 8 == 0 && p.ys[2] % 8 == 0 &&
                  p.ys[0] % 8 == 0;
    if (p.dtype == GCONV_BF16) return dwtcl_launch_t<__nv_bfloat16>(p, q, s, g);
    return dwtcl_launch_t<__half>(p, q, s, g);
}

}  // namespace

const Schedule kDwTcl = {"dw_tcl", dwtcl_supports, dwtcl_launch};

}  // namespace gconv
