// k_row8.cuh -- dw_row8: channels-last depthwise (multiplier 1) whose input
// window slides through registers (executorch PR #25085, description,
// second paragraph, names this schedule for inputs whose channels are
// contiguous).
//
// Design for sm_103a (one persistent pass over HBM):
//  - Work is a flat list of output rows u = ((n*CC + cc)*HC + hc)*OH + oh
//    (image, column chunk, channel chunk, output row).  Each CTA takes one
//    contiguous range of it, so every SM gets the same number of rows to
//    within one.  A run is a maximal range of those rows with one
//    (n, cc, hc); rows oh_a..oh_b of a run read the consecutive input rows
//    oh_a*S_H - pad .. oh_b*S_H - pad + KH - 1, each exactly once.
//  - Input rows stream through a ring of NS shared-memory stages filled by
//    TMA: one thread arms a stage's mbarrier and issues a tiled bulk copy of
//    the row segment (Win pixels x the chunk's channels); the tensor map's
//    out-of-bounds zero fill supplies the padding.  NS rows are in flight;
//    one block barrier per input row frees the stage just read, which the
//    same thread refills at once.  Consumers wait on the stage's barrier
//    phase with a bounded poll.
//  - Thread (cv, pg) owns VEC consecutive channels and S consecutive output
//    pixels.  Its KH*KW weights (fp32 channel pairs) stay in registers for
//    the CTA's lifetime.  Each staged input row is widened once into a
//    window of (S-1)*S_W + KW vectors (32-bit shared addressing) and
//    multiplied (packed fma.rn.f32x2 over channel pairs) into every output
//    row still open on it: R = ceil(((KH - 1)*d + 1) / S_H) (d: dilation,
//    1, or 2 for 3x3 kernels at stride 1; taps then read every d-th row and
//    window slot)
//    accumulator sets rotate through the output rows, with set indices fixed
//    at compile time by unrolling the row loop over one rotation period.
//  - Accumulators start at the bias (fp32); a finished output row is
//    rounded once to the output dtype and stored with coalesced 4/8/16-byte
//    stores through a pointer that advances one output row at a time.
//  - A wait that gives up (it should never happen) poisons the waiting
//    thread's accumulators and bias with NaN and marks the CTA failed: no
//    box is issued or waited for after that, every thread poisons its own
//    accumulators at its next stage, so the outputs are NaN (the failure is
//    visible in the result instead of hanging the GPU, and the store path
//    carries no per-value check); before exiting, the issuing thread waits
//    once more (bounded) for every box it issued that was not seen to arrive.
#pragma once

#include "gconv_internal.h"
#include "launch.cuh"
#include "stencil_math.cuh"
#include "tma.cuh"

#include <type_traits>

namespace gconv {

// Channels per thread: the widest vector (<= 16 bytes) whose KH*KW fp32
// weight pairs fit in about 100 registers.
template <typename T>
constexpr int row8_vec(int K) {
    return K <= 3 ? 4 : 2;
}
// Output pixels per thread and the CTA size cap, which sets how many
// registers a thread may use (weights + R*S accumulator pairs + window).
constexpr int row8_s(int K) { return K == 5 ? 4 : 2; }
constexpr int row8_max_threads(int K) { return K <= 3 ? 256 : (K <= 5 ? 384 : 336); }
// Persistent CTAs per SM (their shared memory splits the SM's).  Measured on
// the 3x3 layers: two 256-thread CTAs overlap one another's barrier and
// wait phases and beat one 512-thread CTA; three are slower.
constexpr int row8_ctas_per_sm(int K) { return K <= 3 ? 2 : 1; }
constexpr int kRow8MaxStages = 8;
// Input rows per stage: one rotation period of the accumulator sets.
constexpr int row8_rows_per_stage(int K, int SH) { return SH * ((K + SH - 1) / SH); }

// Host-computed geometry of one launch.
struct Row8Geom {
    int CVc;        // channel vectors per chunk (threads along channels)
    int PG;         // pixel groups per column chunk (threads along columns)
    int OWc;        // output columns per chunk = PG * S
    int CC, HC;     // column chunks, channel chunks
    int Win;        // input pixels per staged row segment (TMA box width)
    int pitch;      // bytes per staged pixel = chunk channels * element size
    int box_bytes;  // bytes one row copy delivers
    int stage;      // bytes per stage (box_bytes rounded up to 128)
    int NS;         // stages in the ring
    int units;      // output rows in the flat list
    int ctas;
};

struct Row8Run {
    int n, cc, hc, oh0, rows, nin;   // nin = input rows the run reads
};

// The run that starts at flat output row u of a CTA whose rows end at o1.
template <int K, int SH>
__device__ __forceinline__ Row8Run row8_run_at(int u, int o1, int OH, int CC, int HC) {
    Row8Run r;
    const int seg = u / OH;
    r.oh0 = u - seg * OH;
    int end = (seg + 1) * OH;
    if (end > o1) end = o1;
    r.rows = end - u;
    r.nin = (r.rows - 1) * SH + K;
    r.hc = seg % HC;
    const int s2 = seg / HC;
    r.cc = s2 % CC;
    r.n = s2 / CC;
    return r;
}

constexpr float kNaN = __builtin_nanf("");

// Floor division and modulo for compile-time constants (may be negative).
constexpr int fdiv(int a, int b) { return (a >= 0) ? a / b : -((-a + b - 1) / b); }
constexpr int fmod_pos(int a, int b) { return ((a % b) + b) % b; }

// Shared-memory vector loads through 32-bit shared addresses.
template <int BYTES> struct Lds;
template <> struct Lds<4> {
    template <typename V> static __device__ __forceinline__ void load(V &v, uint32_t a) {
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v.w[0]) : "r"(a));
    }
};
template <> struct Lds<8> {
    template <typename V> static __device__ __forceinline__ void load(V &v, uint32_t a) {
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.w[0]), "=r"(v.w[1]) : "r"(a));
    }
};
template <> struct Lds<16> {
    template <typename V> static __device__ __forceinline__ void load(V &v, uint32_t a) {
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                     : "r"(a));
    }
};

template <typename T, int K, int SH, int D>
__global__ void __launch_bounds__(row8_max_threads(K), row8_ctas_per_sm(K))
row8_kernel(const __grid_constant__ CUtensorMap xmap, const T *__restrict__ x,
            const T *__restrict__ w, const T *__restrict__ b, T *__restrict__ y, Params p,
            Row8Geom g) {
    // Let the next kernel in the stream start launching; wait for the
    // previous kernel's memory before reading global memory.
    pdl_launch_dependents();
    pdl_wait();
    constexpr int SW = SH;                       // square strides only
    constexpr int VEC = row8_vec<T>(K);
    constexpr int P = VEC / 2;                   // channel pairs per thread
    constexpr int S = row8_s(K);
    constexpr int VB = VEC * (int)sizeof(T);     // bytes per vector
    constexpr int KX = (K - 1) * D + 1;          // input rows (columns) one output spans
    constexpr int R = (KX + SH - 1) / SH;        // output rows open at once
    constexpr int U = SH * R;                    // rotation period = input rows per stage
    constexpr int WIN = (S - 1) * SW + KX;       // input vectors per window
    using V = Vec<T, VEC>;
    using IO = VecIO<VB>;
    extern __shared__ __align__(128) unsigned char row8_ring[];
    (void)x;

    const int t = threadIdx.x;
    const int cvl = t % g.CVc;
    const int pg = t / g.CVc;

    // This CTA's output rows [o0, o1).
    const int per = g.units / g.ctas, extra = g.units % g.ctas;
    const int o0 = blockIdx.x * per + min((int)blockIdx.x, extra);
    const int o1 = o0 + per + ((int)blockIdx.x < extra ? 1 : 0);
    if (o0 >= o1) return;

    const uint32_t ring = smem_addr(row8_ring);
    const uint32_t bars = ring + (uint32_t)(g.NS * g.stage);   // NS mbarriers
    // Set once any wait of the CTA gives up: no box is issued or waited for
    // after it (the stores become NaN).
    volatile int *abort_flag = reinterpret_cast<volatile int *>(row8_ring + g.NS * g.stage + 8 * g.NS);
    // fp32 weights [tap][chunk channel] and bias, after the barriers
    float *wsm = reinterpret_cast<float *>(row8_ring + g.NS * g.stage + 8 * g.NS + 16);
    const int row_bytes = g.Win * g.pitch;       // one staged input row

    // Producer (thread 0 only): the run and stage of the next box.  A stage
    // holds U consecutive input rows of one run.
    Row8Run prun{};
    int pnext_u = 0, pst = 0, pnst = 0, pslot = 0;
    int pissued = 0;       // boxes issued so far
    bool pdone = false;
    auto issue = [&]() {
        if (pdone) return;
        ++pissued;
        const uint32_t bar = bars + 8u * pslot;
        mbar_arrive_expect_tx(bar, (uint32_t)g.box_bytes);
        tma_load_4d(ring + (uint32_t)(pslot * g.stage), &xmap, bar, prun.hc * g.CVc * VEC,
                    prun.cc * g.OWc * SW - p.pbw, prun.oh0 * SH - p.pbh + pst * U, prun.n);
        if (++pslot == g.NS) pslot = 0;
        if (++pst == pnst) {
            if (pnext_u >= o1) {
                pdone = true;
            } else {
                prun = row8_run_at<KX, SH>(pnext_u, o1, p.OH, g.CC, g.HC);
                pnext_u += prun.rows;
                pst = 0;
                pnst = (prun.nin + U - 1) / U;
            }
        }
    };
    float2 wr[K][K][P];
    float2 bias[P];
    // Stage chunk hc's weights and bias through shared memory with coalesced
    // loads ([tap][channel] fp32), then take this thread's channel pairs.
    auto stage_weights = [&](int hc) {
        const int cb = g.CVc * VEC, cfirst = hc * cb;
        constexpr int QW = 8;   // loads in flight per thread before their stores
        for (int e0 = t; e0 < cb * K * K; e0 += QW * blockDim.x) {
            float v[QW];
#pragma unroll
            for (int q = 0; q < QW; ++q) {
                const int e = e0 + q * blockDim.x;
                const int cl = e / (K * K), tap = e - cl * (K * K);
                const int c = cfirst + cl;
                const int kh = tap / K, kw = tap - kh * K;
                v[q] = (e < cb * K * K && c < p.C_out)
                           ? load_f32(w + (int64_t)c * p.ws[0] + kh * p.ws[2] + kw * p.ws[3]) : 0.f;
            }
#pragma unroll
            for (int q = 0; q < QW; ++q) {
                const int e = e0 + q * blockDim.x;
                const int cl = e / (K * K), tap = e - cl * (K * K);
                if (e < cb * K * K) wsm[tap * cb + cl] = v[q];
            }
        }
        for (int cl = t; cl < cb; cl += blockDim.x) {
            const int c = cfirst + cl;
            wsm[K * K * cb + cl] = (c < p.C_out && p.has_bias) ? load_f32(b + (int64_t)c * p.bs) : 0.f;
        }
    };
    auto take_weights = [&]() {
        const int cb = g.CVc * VEC;
        const float2 *src = reinterpret_cast<const float2 *>(wsm) + cvl * P;
#pragma unroll
        for (int kh = 0; kh < K; ++kh)
#pragma unroll
            for (int kw = 0; kw < K; ++kw)
#pragma unroll
                for (int k = 0; k < P; ++k) wr[kh][kw][k] = src[((kh * K + kw) * cb) / 2 + k];
#pragma unroll
        for (int k = 0; k < P; ++k) bias[k] = src[(K * K * cb) / 2 + k];
    };
    // The first run's weights are fetched before the row stream starts:
    // issued behind it they would wait for it.
    int loaded_hc = row8_run_at<KX, SH>(o0, o1, p.OH, g.CC, g.HC).hc;
    stage_weights(loaded_hc);

    if (t == 0) {
        tma_prefetch_map(&xmap);
        for (int i = 0; i < g.NS; ++i) mbar_init(bars + 8u * i, 1);
        *abort_flag = 0;
        fence_barrier_init();
        prun = row8_run_at<KX, SH>(o0, o1, p.OH, g.CC, g.HC);
        pnext_u = o0 + prun.rows;
        pnst = (prun.nin + U - 1) / U;
        for (int i = 0; i < g.NS; ++i) issue();   // prologue: NS stages in flight
    }
    __syncthreads();
    take_weights();

    int cslot = 0;        // stage of the consumer's next box
    uint32_t cphase = 0;  // parity of that stage's current use

    bool bad = false;     // a box wait gave up (outputs become NaN)
    int cwaited = 0;      // boxes this thread has seen arrive
    int u = o0;
    while (u < o1) {
        const Row8Run run = row8_run_at<KX, SH>(u, o1, p.OH, g.CC, g.HC);
        u += run.rows;
        const int c0 = (run.hc * g.CVc + cvl) * VEC;
        const bool active = c0 < p.C_out;
        if (run.hc != loaded_hc) {
            loaded_hc = run.hc;
            __syncthreads();
            stage_weights(loaded_hc);
            __syncthreads();
            take_weights();
            if (bad)
#pragma unroll
                for (int k = 0; k < P; ++k) bias[k] = make_float2(kNaN, kNaN);
        }
        // Accumulator set s serves the output rows j with j mod R == s; it
        // is reset to the bias right after its row's last input row.
        float2 acc[R][S][P];
#pragma unroll
        for (int s = 0; s < R; ++s)
#pragma unroll
            for (int i = 0; i < S; ++i)
#pragma unroll
                for (int k = 0; k < P; ++k) acc[s][i][k] = bias[k];

        const int ow0 = run.cc * g.OWc + pg * S;
        // output row r0 / SH of the run at this thread's pixels and channels
        T *ystage = y + (int64_t)run.n * p.ys[0] + (int64_t)run.oh0 * p.ys[2] +
                    (int64_t)ow0 * p.ys[3] + (active ? c0 : 0);
        bool pix_ok[S];
#pragma unroll
        for (int i = 0; i < S; ++i) pix_ok[i] = ow0 + i < p.OW;
        const uint32_t win0 = ring + (uint32_t)(cvl * VB + pg * S * SW * g.pitch);

        for (int r0 = 0; r0 < run.nin; r0 += U) {
            const bool arrived = !bad && mbar_wait(bars + 8u * cslot, cphase, abort_flag);
            if (arrived) ++cwaited;
            // Thread 0 reads the flag here, off the refill's critical path: a
            // failure seen one stage late costs one more box, drained below.
            if (t == 0 && *abort_flag) pdone = true;
            if (!arrived && !bad) {
                // The box did not arrive (or another thread's did not): poison
                // every open accumulator and the bias, so every output this
                // thread stores from now on is NaN (the bias is poisoned
                // again after a weight reload), and stop the ring.
                bad = true;
                *abort_flag = 1;
#pragma unroll
                for (int s = 0; s < R; ++s)
#pragma unroll
                    for (int i = 0; i < S; ++i)
#pragma unroll
                        for (int k = 0; k < P; ++k) acc[s][i][k] = make_float2(kNaN, kNaN);
#pragma unroll
                for (int k = 0; k < P; ++k) bias[k] = make_float2(kNaN, kNaN);
            }
            const uint32_t stage0 = win0 + (uint32_t)(cslot * g.stage);
            // Straight-line over the stage's U rows (no branches around the
            // arithmetic, so the scheduler can overlap the rows' loads):
            // every row is multiplied into every set it feeds; each set is
            // reset right after its last tap row.  MODE 1 is the run's first
            // stage and MODE 2 a stage that starts at the run's end: their
            // taps that feed output rows before the run (MODE 1) or past it
            // (MODE 2) are left out at compile time; the other stages have
            // none, and sets whose output row lies outside the run are never
            // stored.
            auto stage_body = [&](auto mode) {
                constexpr int MODE = decltype(mode)::value;
#pragma unroll
                for (int ph = 0; ph < U; ++ph) {
                    const int r = r0 + ph;
                    const uint32_t st = stage0 + (uint32_t)(ph * row_bytes);
                    float2 xr[WIN][P];
#pragma unroll
                    for (int j = 0; j < WIN; ++j) {
                        V v;
                        Lds<VB>::load(v, st + (uint32_t)(j * g.pitch));
                        widen<T, VEC>(v, xr[j]);
                    }
#pragma unroll
                    for (int kh = 0; kh < K; ++kh) {
                        const int d = ph - kh * D;           // (r - kh*D) - r0
                        if (fmod_pos(d, SH) != 0) continue;  // no output row has tap row kh here
                        if (MODE == 1 && d < 0) continue;    // its output row precedes the run
                        if (MODE == 2 && d >= 0) continue;   // its output row is past the run
                        const int set = fmod_pos(fdiv(d, SH), R);
#pragma unroll
                        for (int i = 0; i < S; ++i)
#pragma unroll
                            for (int kw = 0; kw < K; ++kw)
#pragma unroll
                                for (int k = 0; k < P; ++k)   // packed: half the issue slots
                                    fma2_packed(acc[set][i][k], wr[kh][kw][k], xr[i * SW + kw * D][k]);
                    }
                    // The output row whose last tap row this was is done.
                    const int d = ph - (KX - 1);
                    if (fmod_pos(d, SH) == 0) {
                        const int set = fmod_pos(fdiv(d, SH), R);
                        const int jn = r - (KX - 1);         // SH * output row within the run
                        if (active && jn >= 0 && jn < run.rows * SH) {
                            // output row jn / SH = r0 / SH + (ph - K + 1) / SH
                            T *yrow = ystage + (int64_t)fdiv(ph - (KX - 1), SH) * p.ys[2];
#pragma unroll
                            for (int i = 0; i < S; ++i)
                                if (pix_ok[i])
                                    IO::store(yrow + (int64_t)i * p.ys[3], pack_pairs<T, VEC>(acc[set][i]));
                        }
#pragma unroll
                        for (int i = 0; i < S; ++i)
#pragma unroll
                            for (int k = 0; k < P; ++k) acc[set][i][k] = bias[k];
                    }
                }
            };
            if (r0 == 0)
                stage_body(std::integral_constant<int, 1>{});
            else if (r0 == run.rows * SH)
                stage_body(std::integral_constant<int, 2>{});
            else
                stage_body(std::integral_constant<int, 0>{});
            ystage += (int64_t)R * p.ys[2];   // U / SH output rows per stage
            if (++cslot == g.NS) {
                cslot = 0;
                cphase ^= 1u;
            }
            __syncthreads();          // every thread is done with that stage
            if (t == 0) issue();      // refill it with the box NS stages ahead
        }
    }
    // After a failed wait, boxes issued but never seen to arrive may still be
    // landing in this CTA's shared memory: wait for each once more (bounded)
    // before the CTA exits.  Issue and arrival follow the same slot order.
    if (t == 0 && *abort_flag)
        for (int q = cwaited; q < pissued; ++q)
            (void)mbar_wait(bars + 8u * (uint32_t)(q % g.NS), (uint32_t)((q / g.NS) & 1));
}

// Launch geometry for one call; false when the shape does not fit.
template <typename T, int K>
bool row8_geometry(const Params &p, Row8Geom &g) {
    constexpr int VEC = row8_vec<T>(K);
    constexpr int S = row8_s(K);
    constexpr int VB = VEC * (int)sizeof(T);
    constexpr int MAXT = row8_max_threads(K);
    if (p.C_out % VEC != 0) return false;
    const int CV = p.C_out / VEC;
    int cv_cap = MAXT < 256 / VEC ? MAXT : 256 / VEC;   // TMA box: <= 256 channels
    g.CVc = CV < cv_cap ? CV : cv_cap;
    if ((g.CVc * VB) % 16 != 0) return false;            // box rows of whole 16-byte units
    g.HC = (CV + g.CVc - 1) / g.CVc;
    const int pg_max = MAXT / g.CVc;
    const int pg_need = (p.OW + S - 1) / S;
    const int KX = (K - 1) * p.dw + 1;   // columns (rows: dh) one output spans
    // Split the columns evenly over the fewest chunks that fit the CTA and
    // keep each staged segment within the 256-pixel TMA box.
    int cc = (pg_need + pg_max - 1) / pg_max;
    for (;; ++cc) {
        const int pg = (pg_need + cc - 1) / cc;
        if ((pg * S - 1) * p.sw + KX <= 256) break;
    }
    g.PG = (pg_need + cc - 1) / cc;
    g.OWc = g.PG * S;
    g.CC = (p.OW + g.OWc - 1) / g.OWc;
    g.Win = (g.OWc - 1) * p.sw + KX;
    g.pitch = g.CVc * VB;
    g.box_bytes = g.Win * g.pitch * row8_rows_per_stage((K - 1) * p.dh + 1, p.sh);
    g.stage = (g.box_bytes + 127) / 128 * 128;
    int ns = (200 * 1024 / row8_ctas_per_sm(K) - (K * K + 1) * g.CVc * VEC * 4) / g.stage;
    if (ns > kRow8MaxStages) ns = kRow8MaxStages;
    if (ns < 2) return false;
    g.NS = ns;
    const int64_t units = (int64_t)p.N * g.CC * g.HC * p.OH;
    if (units > INT32_MAX / 2) return false;
    g.units = (int)units;
    const int cap = 152 * row8_ctas_per_sm(K);   // persistent CTAs
    g.ctas = g.units < cap ? g.units : cap;
    return true;
}

template <typename T, int K, int SH, int D>
cudaError_t row8_launch_t(const Params &p, const Ptrs &q, cudaStream_t s) {
    constexpr int VEC = row8_vec<T>(K);
    Row8Geom g;
    if (!row8_geometry<T, K>(p, g)) return cudaErrorNotSupported;
    // x as (C, W, H, N), innermost first; a box is one row segment.
    const uint64_t es = sizeof(T);
    const uint64_t dims[4] = {(uint64_t)p.C_out, (uint64_t)p.W, (uint64_t)p.H, (uint64_t)p.N};
    const uint64_t strides[3] = {(uint64_t)p.xs[3] * es, (uint64_t)p.xs[2] * es,
                                 (uint64_t)p.xs[0] * es};
    const uint32_t box[4] = {(uint32_t)(g.CVc * VEC), (uint32_t)g.Win,
                             (uint32_t)row8_rows_per_stage((K - 1) * D + 1, SH), 1u};
    CUtensorMap map;
    if (!tma_encode_4d(&map, tma_dtype<T>(), q.x, dims, strides, box)) return cudaErrorInvalidValue;
    const size_t smem = (size_t)g.NS * g.stage + 8 * (size_t)g.NS + 16 +
                        (size_t)(K * K + 1) * g.CVc * VEC * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(row8_kernel<T, K, SH, D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_kernel(row8_kernel<T, K, SH, D>, dim3(g.ctas), dim3(g.CVc * g.PG), smem, s, map,
                   static_cast<const T *>(q.x), static_cast<const T *>(q.w),
                   static_cast<const T *>(q.b), static_cast<T *>(q.y), p, g);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename T>
cudaError_t row8_launch_dtype(const Params &p, const Ptrs &q, cudaStream_t s) {
    const int K = p.KH, SH = p.sh;
#define GCONV_ROW8_CASE(KK, SS, DD) \
    if (K == KK && SH == SS && p.dh == DD) return row8_launch_t<T, KK, SS, DD>(p, q, s);
    GCONV_ROW8_CASE(3, 1, 1) GCONV_ROW8_CASE(3, 2, 1)
    GCONV_ROW8_CASE(5, 1, 1) GCONV_ROW8_CASE(5, 2, 1)
    GCONV_ROW8_CASE(7, 1, 1) GCONV_ROW8_CASE(7, 2, 1)
    GCONV_ROW8_CASE(3, 1, 2)
#undef GCONV_ROW8_CASE
    return cudaErrorNotSupported;
}

template <typename T>
bool row8_fits_dtype(const Params &p) {
    Row8Geom g;
    switch (p.KH) {
    case 3: return row8_geometry<T, 3>(p, g);
    case 5: return row8_geometry<T, 5>(p, g);
    case 7: return row8_geometry<T, 7>(p, g);
    }
    return false;
}

cudaError_t row8_launch_f32(const Params &p, const Ptrs &q, cudaStream_t s);
cudaError_t row8_launch_f16(const Params &p, const Ptrs &q, cudaStream_t s);
cudaError_t row8_launch_bf16(const Params &p, const Ptrs &q, cudaStream_t s);

}  // namespace gconv
