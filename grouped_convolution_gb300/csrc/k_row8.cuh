// k_row8.cuh -- dw_row8: channels-last depthwise (multiplier 1) with a
// register sliding window (executorch PR #25085, description, second
// paragraph: "a register sliding window for channel-contiguous inputs").
//
// Design for sm_103a (one persistent pass over HBM):
//  - Work is a flat list of output rows u = ((n*CC + cc)*HC + hc)*OH + oh
//    (image, column chunk, channel chunk, output row).  Each CTA takes one
//    contiguous range of it, so every SM gets the same number of rows to
//    within one.  A run is a maximal range of those rows with one
//    (n, cc, hc); rows oh_a..oh_b of a run read the consecutive input rows
//    oh_a*S_H - pad .. oh_b*S_H - pad + KH - 1, each exactly once.
//  - Input rows stream through a ring of NS shared-memory stages with
//    16-byte cp.async copies issued by all threads; zero-fill supplies the
//    padding, so no bounds test remains in the arithmetic.  NS - 1 rows are
//    in flight; one block barrier per input row both publishes the row and
//    frees the stage read one row earlier, which is refilled at once.
//  - Thread (cv, pg) owns VEC consecutive channels and S consecutive output
//    pixels.  Its KH*KW weights (fp32 channel pairs) stay in registers for
//    the CTA's lifetime.  Each staged input row is widened once into a
//    window of (S-1)*S_W + KW vectors and multiplied into every output row
//    still open on it: R = ceil(KH / S_H) accumulator sets rotate through
//    the output rows, with set indices fixed at compile time by unrolling
//    the row loop over one rotation period.
//  - Accumulators start at the bias (fp32); a finished output row is
//    rounded once to the output dtype and stored with coalesced 4/8/16-byte
//    stores.
//  - No spin waits: the only waits are cp.async.wait_group on the thread's
//    own copies and block barriers.
#pragma once

#include "gconv_internal.h"
#include "stencil_math.cuh"

namespace gconv {

// Channels per thread: the widest vector (<= 16 bytes) whose KH*KW fp32
// weight pairs fit in about 100 registers.
template <typename T>
constexpr int row8_vec(int K) {
    return K <= 3 ? (sizeof(T) == 4 ? 4 : 8) : 2;
}
// Output pixels per thread and the CTA size cap, which sets how many
// registers a thread may use (weights + R*S accumulator pairs + window).
constexpr int row8_s(int K) { return K == 5 ? 4 : 2; }
constexpr int row8_max_threads(int K) { return K <= 3 ? 256 : (K <= 5 ? 448 : 336); }
constexpr int kRow8Stages = 6;          // ring depth: 5 input rows in flight

// Host-computed geometry of one launch.
struct Row8Geom {
    int CVc;        // channel vectors per chunk (threads along channels)
    int PG;         // pixel groups per column chunk (threads along columns)
    int OWc;        // output columns per chunk = PG * S
    int CC, HC;     // column chunks, channel chunks
    int Win;        // input pixels per staged row segment
    int pitch;      // bytes per staged pixel (multiple of 16)
    int stage;      // bytes per stage
    int chunk16;    // 16-byte copies per staged pixel
    int units;      // output rows in the flat list
    int ctas;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                 "r"(bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// A run: output rows [oh0, oh0 + rows) of one (n, cc, hc).
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

// Floor division and modulo for compile-time constants (may be negative).
constexpr int fdiv(int a, int b) { return (a >= 0) ? a / b : -((-a + b - 1) / b); }
constexpr int fmod_pos(int a, int b) { return ((a % b) + b) % b; }

template <typename T, int K, int SH>
__global__ void __launch_bounds__(row8_max_threads(K), 1)
row8_kernel(const T *__restrict__ x, const T *__restrict__ w, const T *__restrict__ b,
            T *__restrict__ y, Params p, Row8Geom g) {
    constexpr int SW = SH;                       // square strides only
    constexpr int VEC = row8_vec<T>(K);
    constexpr int P = VEC / 2;                   // channel pairs per thread
    constexpr int S = row8_s(K);
    constexpr int VB = VEC * (int)sizeof(T);     // bytes per vector
    constexpr int R = (K + SH - 1) / SH;         // output rows open at once
    constexpr int U = SH * R;                    // rotation period of the sets
    constexpr int WIN = (S - 1) * SW + K;        // input vectors per window
    constexpr int NS = kRow8Stages;
    using V = Vec<T, VEC>;
    using IO = VecIO<VB>;
    extern __shared__ __align__(16) unsigned char row8_ring[];

    const int t = threadIdx.x;
    const int nthreads = g.CVc * g.PG;
    const int cvl = t % g.CVc;
    const int pg = t / g.CVc;

    // This CTA's output rows [o0, o1).
    const int per = g.units / g.ctas, extra = g.units % g.ctas;
    const int o0 = blockIdx.x * per + min((int)blockIdx.x, extra);
    const int o1 = o0 + per + ((int)blockIdx.x < extra ? 1 : 0);
    if (o0 >= o1) return;

    const uint32_t ring = (uint32_t)__cvta_generic_to_shared(row8_ring);
    const int c_bytes = p.C_out * (int)sizeof(T);

    const int64_t xs3b = p.xs[3] * (int64_t)sizeof(T);
    // This thread's first 16-byte copy of a stage and the step between its
    // copies (copy q = t + i * nthreads covers pixel q / chunk16).
    const int cp_pix0 = t / g.chunk16, cp_sub0 = t - cp_pix0 * g.chunk16;
    const int cp_dpix = nthreads / g.chunk16, cp_dsub = nthreads - cp_dpix * g.chunk16;

    // Producer state: the run and input row of the next entry to issue.
    Row8Run prun = row8_run_at<K, SH>(o0, o1, p.OH, g.CC, g.HC);
    int pnext_u = o0 + prun.rows;
    int pr = 0;
    bool pdone = false;
    int pslot = 0;

    // Copy the producer's next input row into its stage (nothing once the
    // list is exhausted) and commit one group, so group counts stay uniform.
    auto issue = [&]() {
        if (!pdone) {
            const int ih = prun.oh0 * SH - p.pbh + pr;
            const bool row_ok = ih >= 0 && ih < p.H;
            const int iw_start = prun.cc * g.OWc * SW - p.pbw;
            const int cb0 = prun.hc * g.CVc * VB;
            const uint32_t dst0 = ring + (uint32_t)(pslot * g.stage);
            const char *src_row =
                reinterpret_cast<const char *>(x + (int64_t)prun.n * p.xs[0] +
                                               (int64_t)(row_ok ? ih : 0) * p.xs[2]) + cb0;
            int pix = cp_pix0, sub = cp_sub0;
            while (pix < g.Win) {
                const int iw = iw_start + pix;
                const int cbyte = sub * 16;
                int bytes = c_bytes - (cb0 + cbyte);
                bytes = bytes > 16 ? 16 : bytes;
                const bool ok = row_ok && iw >= 0 && iw < p.W && bytes > 0;
                const char *src = ok ? src_row + (int64_t)iw * xs3b + cbyte
                                     : reinterpret_cast<const char *>(x);
                cp_async16(dst0 + (uint32_t)(pix * g.pitch + cbyte), src, ok ? bytes : 0);
                pix += cp_dpix;
                sub += cp_dsub;
                if (sub >= g.chunk16) { sub -= g.chunk16; ++pix; }
            }
            if (++pr == prun.nin) {
                if (pnext_u >= o1) {
                    pdone = true;
                } else {
                    prun = row8_run_at<K, SH>(pnext_u, o1, p.OH, g.CC, g.HC);
                    pnext_u += prun.rows;
                    pr = 0;
                }
            }
        }
        cp_async_commit();
        if (++pslot == NS) pslot = 0;
    };

#pragma unroll 1
    for (int i = 0; i < NS - 1; ++i) issue();   // prologue: NS - 1 rows in flight

    float2 wr[K][K][P];
    float2 bias[P];
    int loaded_hc = -1;
    int cslot = 0;                  // stage of the consumer's next input row

    int u = o0;
    while (u < o1) {
        const Row8Run run = row8_run_at<K, SH>(u, o1, p.OH, g.CC, g.HC);
        u += run.rows;
        const int c0 = (run.hc * g.CVc + cvl) * VEC;
        const bool active = c0 < p.C_out;
        if (run.hc != loaded_hc) {
            loaded_hc = run.hc;
#pragma unroll
            for (int kh = 0; kh < K; ++kh)
#pragma unroll
                for (int kw = 0; kw < K; ++kw)
#pragma unroll
                    for (int k = 0; k < P; ++k) {
                        const T *wp = w + (int64_t)(c0 + 2 * k) * p.ws[0] + kh * p.ws[2] +
                                      kw * p.ws[3];
                        wr[kh][kw][k] = active ? make_float2(load_f32(wp), load_f32(wp + p.ws[0]))
                                               : make_float2(0.f, 0.f);
                    }
#pragma unroll
            for (int k = 0; k < P; ++k)
                bias[k] = (active && p.has_bias)
                              ? make_float2(load_f32(b + (int64_t)(c0 + 2 * k) * p.bs),
                                            load_f32(b + (int64_t)(c0 + 2 * k + 1) * p.bs))
                              : make_float2(0.f, 0.f);
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
        T *ybase = y + (int64_t)run.n * p.ys[0] + (int64_t)ow0 * p.ys[3] + c0;
        const unsigned char *win0 = row8_ring + cvl * VB + pg * S * SW * g.pitch;

        for (int r0 = 0; r0 < run.nin; r0 += U) {
#pragma unroll
            for (int ph = 0; ph < U; ++ph) {
                const int r = r0 + ph;
                if (r < run.nin) {
                    // Input row r: complete for this thread, then for all; the
                    // stage read one row ago is free and is refilled at once.
                    cp_async_wait<NS - 2>();
                    __syncthreads();
                    issue();
                    if (active) {
                        const unsigned char *st = win0 + cslot * g.stage;
                        float2 xr[WIN][P];
#pragma unroll
                        for (int j = 0; j < WIN; ++j) {
                            V v;
                            IO::load_shared(v, st + j * g.pitch);
                            widen<T, VEC>(v, xr[j]);
                        }
#pragma unroll
                        for (int kh = 0; kh < K; ++kh) {
                            const int d = ph - kh;               // (r - kh) - r0
                            if (fmod_pos(d, SH) != 0) continue;  // no output row has tap row kh here
                            const int set = fmod_pos(fdiv(d, SH), R);
                            const int jn = r - kh;   // SH * (output row within the run)
                            if (jn >= 0 && jn < run.rows * SH) {
#pragma unroll
                                for (int i = 0; i < S; ++i)
#pragma unroll
                                    for (int kw = 0; kw < K; ++kw)
#pragma unroll
                                        for (int k = 0; k < P; ++k)
                                            fma2(acc[set][i][k], wr[kh][kw][k], xr[i * SW + kw][k]);
                            }
                        }
                        // The output row whose last tap row this was is done.
                        {
                            const int d = ph - (K - 1);
                            if (fmod_pos(d, SH) == 0) {
                                const int set = fmod_pos(fdiv(d, SH), R);
                                const int jn = r - (K - 1);
                                if (jn >= 0) {
                                    T *yrow = ybase + (int64_t)(run.oh0 + jn / SH) * p.ys[2];
#pragma unroll
                                    for (int i = 0; i < S; ++i)
                                        if (ow0 + i < p.OW)
                                            IO::store(yrow + (int64_t)i * p.ys[3],
                                                      pack_pairs<T, VEC>(acc[set][i]));
                                }
#pragma unroll
                                for (int i = 0; i < S; ++i)
#pragma unroll
                                    for (int k = 0; k < P; ++k) acc[set][i][k] = bias[k];
                            }
                        }
                    }
                    if (++cslot == NS) cslot = 0;
                }
            }
        }
    }
    cp_async_wait<0>();
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
    g.CVc = CV < MAXT ? CV : MAXT;
    g.HC = (CV + g.CVc - 1) / g.CVc;
    const int pg_max = MAXT / g.CVc;
    const int pg_need = (p.OW + S - 1) / S;
    // Split the columns evenly over the fewest chunks that fit the CTA.
    const int cc = (pg_need + pg_max - 1) / pg_max;
    g.PG = (pg_need + cc - 1) / cc;
    g.OWc = g.PG * S;
    g.CC = (p.OW + g.OWc - 1) / g.OWc;
    g.Win = (g.OWc - 1) * p.sw + K;
    g.chunk16 = (g.CVc * VB + 15) / 16;
    g.pitch = g.chunk16 * 16;
    g.stage = g.Win * g.pitch;
    if ((size_t)g.stage * kRow8Stages > 220 * 1024) return false;
    // byte offsets within one image row fit in 32 bits
    if ((int64_t)p.W * p.xs[3] * (int64_t)sizeof(T) + p.C_out * (int64_t)sizeof(T) > INT32_MAX)
        return false;
    const int64_t units = (int64_t)p.N * g.CC * g.HC * p.OH;
    if (units > INT32_MAX / 2) return false;
    g.units = (int)units;
    g.ctas = g.units < 152 ? g.units : 152;   // one persistent CTA per SM
    return true;
}

template <typename T, int K, int SH>
cudaError_t row8_launch_t(const Params &p, const Ptrs &q, cudaStream_t s) {
    Row8Geom g;
    if (!row8_geometry<T, K>(p, g)) return cudaErrorNotSupported;
    const size_t smem = (size_t)kRow8Stages * g.stage;
    cudaError_t e = cudaFuncSetAttribute(row8_kernel<T, K, SH>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    row8_kernel<T, K, SH><<<g.ctas, g.CVc * g.PG, smem, s>>>(
        static_cast<const T *>(q.x), static_cast<const T *>(q.w), static_cast<const T *>(q.b),
        static_cast<T *>(q.y), p, g);
    return cudaGetLastError();
}

template <typename T>
cudaError_t row8_launch_dtype(const Params &p, const Ptrs &q, cudaStream_t s) {
    const int K = p.KH, SH = p.sh;
#define GCONV_ROW8_CASE(KK, SS) \
    if (K == KK && SH == SS) return row8_launch_t<T, KK, SS>(p, q, s);
    GCONV_ROW8_CASE(3, 1) GCONV_ROW8_CASE(3, 2)
    GCONV_ROW8_CASE(5, 1) GCONV_ROW8_CASE(5, 2)
    GCONV_ROW8_CASE(7, 1) GCONV_ROW8_CASE(7, 2)
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
