// k_row8t.cuh -- dw_row8's transposed form: channels-last depthwise
// transposed convolution (one input and one output channel per group) at
// stride 2 in both dims with a square 3x3, 5x5 or 7x7 kernel, dilation 1.
// Output o reads input (o + pad_before - k) / 2 where that is a whole number
// inside the input (executorch PR #25091 "Run transposed convolutions on the
// implicit-GEMM template", description, second paragraph).  This is the
// input gradient of a stride-2 depthwise convolution, and 2x upsampling.
//
// Design (a gather over a ring of input rows):
//  - Work is a flat list of output rows u = ((n*CC + cc)*HC + hc)*OH + oh,
//    split evenly over persistent CTAs; a run is a maximal range of rows of
//    one (n, cc, hc).
//  - The input rows a run reads, j = floor((oh_first + pad - (K-1))/2) ..
//    floor((oh_last + pad)/2), stream through a ring of NS shared-memory
//    stages, one row segment per stage (a TMA box; its zero fill supplies the
//    rows and columns outside the input), each read once from HBM.
//  - Output rows go in pairs (r, r + 1) with r + pad even: row r takes the
//    even taps kh = 2a and row r + 1 the odd ones kh = 2a + 1, both from
//    input row (r + pad)/2 - a, so a pair reads ceil(K/2) input rows, all in
//    the ring, each window loaded once for both rows.  A row is released, and
//    its stage refilled, once no later pair of the run reads it; one block
//    barrier per pair.
//  - Thread (cv, pg) owns VEC channels and S = 4 consecutive output columns
//    starting at an even distance from -pad_w (a chunk starts one column to
//    the left when pad_w is odd; that column is not stored), so which taps an
//    output takes and where they sit is fixed at compile time: output i at
//    tap kw (i - kw even) reads slot (i - kw + K - 1)/2 of a window of
//    (S + K - 2)/2 + 1 input vectors, loaded and widened once per input row.
//  - Weights and bias in fp32 registers, packed FMAs over channel pairs, one
//    rounding per output, vector stores.
//  - Bounded waits as in the forward: a wait that gives up makes the thread's
//    outputs NaN and stops the ring; before exiting, the issuing thread waits
//    once more (bounded) for every box it issued that was not seen to arrive.
#pragma once

#include "k_row8.cuh"

namespace gconv {

constexpr int kRowTS = 4;   // output columns per thread (even)

// CTA size cap and persistent CTAs per SM.  3x3, measured on six shapes:
// four 128-thread CTAs per SM beat two of 256 by 4-11 % and three of 160
// (more CTAs overlap one another's per-pair barriers); 5x5 and 7x7 keep the
// forward's shape.
constexpr int rowt_max_threads(int K) { return K == 3 ? 128 : row8_max_threads(K); }
constexpr int rowt_ctas_per_sm(int K) { return K == 3 ? 4 : row8_ctas_per_sm(K); }

constexpr int rowt_win(int K) { return (kRowTS + K - 2) / 2 + 1; }

struct RowTGeom {
    int CVc, HC;     // channel vectors per chunk, channel chunks
    int PG;          // pixel groups per column chunk
    int OWc;         // output columns per chunk = PG * S
    int CC;          // column chunks
    int sh0;         // pad_w & 1: chunks start that many columns left of 0
    int Wq;          // input columns per staged segment (TMA box width)
    int pitch;       // bytes per staged pixel
    int box_bytes;   // bytes one row copy delivers
    int stage;       // bytes per stage (rounded up to 128)
    int NS;          // stages (a power of two)
    int ns_log2;
    int units, ctas;
};

struct RowTRun {
    int n, cc, hc, oh0, rows;
    int j0, nj;      // first input row the run reads, and how many
};

__device__ __forceinline__ RowTRun rowt_run_at(int u, int o1, const Params &p,
                                               const RowTGeom &g, int K) {
    RowTRun r;
    const int seg = u / p.OH;
    r.oh0 = u - seg * p.OH;
    int end = (seg + 1) * p.OH;
    if (end > o1) end = o1;
    r.rows = end - u;
    r.hc = seg % g.HC;
    const int s2 = seg / g.HC;
    r.cc = s2 % g.CC;
    r.n = s2 / g.CC;
    r.j0 = (r.oh0 + p.pbh - (K - 1)) >> 1;             // floor
    const int j1 = (r.oh0 + r.rows - 1 + p.pbh) >> 1;  // floor
    r.nj = j1 - r.j0 + 1;
    return r;
}

template <typename T, int K>
bool rowt_geometry(const Params &p, RowTGeom &g) {
    constexpr int VEC = row8_vec<T>(K);
    constexpr int S = kRowTS;
    constexpr int VB = VEC * (int)sizeof(T);
    constexpr int MAXT = rowt_max_threads(K);
    constexpr int WIN = rowt_win(K);
    if (p.C_out % VEC != 0) return false;
    const int CV = p.C_out / VEC;
    const int cv_cap = MAXT < 256 / VEC ? MAXT : 256 / VEC;   // TMA box: <= 256 channels
    g.CVc = CV < cv_cap ? CV : cv_cap;
    if ((g.CVc * VB) % 16 != 0) return false;
    g.HC = (CV + g.CVc - 1) / g.CVc;
    g.sh0 = p.pbw & 1;
    const int cols = p.OW + g.sh0;
    const int pg_max = MAXT / g.CVc;
    const int pg_need = (cols + S - 1) / S;
    int cc = (pg_need + pg_max - 1) / pg_max;
    for (;; ++cc) {
        const int pg = (pg_need + cc - 1) / cc;
        if ((pg - 1) * (S / 2) + WIN <= 256) break;
    }
    g.PG = (pg_need + cc - 1) / cc;
    g.OWc = g.PG * S;
    g.CC = (cols + g.OWc - 1) / g.OWc;
    g.Wq = (g.PG - 1) * (S / 2) + WIN;
    g.pitch = g.CVc * VB;
    g.box_bytes = g.Wq * g.pitch;
    g.stage = (g.box_bytes + 127) / 128 * 128;
    // A power of two, so slots and phases come from masks and shifts.
    const int fit = (200 * 1024 / rowt_ctas_per_sm(K) - 8 * kRow8MaxStages - 16) / g.stage;
    int ns = kRow8MaxStages, l2 = 3;
    while (ns > fit) {
        ns >>= 1;
        --l2;
    }
    if (ns < (K + 1) / 2 + 2) return false;
    g.NS = ns;
    g.ns_log2 = l2;
    const int64_t units = (int64_t)p.N * g.CC * g.HC * p.OH;
    if (units > INT32_MAX / 2) return false;
    g.units = (int)units;
    const int cap = 152 * rowt_ctas_per_sm(K);
    g.ctas = g.units < cap ? g.units : cap;
    return true;
}

template <typename T, int K>
__global__ void __launch_bounds__(rowt_max_threads(K), rowt_ctas_per_sm(K))
row8t_kernel(const __grid_constant__ CUtensorMap xmap, const T *__restrict__ w,
             const T *__restrict__ b, T *__restrict__ y, Params p, RowTGeom g) {
    pdl_launch_dependents();
    pdl_wait();
    constexpr int VEC = row8_vec<T>(K);
    constexpr int P = VEC / 2;
    constexpr int S = kRowTS;
    constexpr int VB = VEC * (int)sizeof(T);
    constexpr int WIN = rowt_win(K);
    constexpr int KE = K - 1;   // K is odd
    using V = Vec<T, VEC>;
    using IO = VecIO<VB>;
    extern __shared__ __align__(128) unsigned char rowt_ring[];

    const int t = threadIdx.x;
    const int cvl = t % g.CVc;
    const int pg = t / g.CVc;

    const int per = g.units / (int)gridDim.x, extra = g.units % (int)gridDim.x;
    const int o0 = (int)blockIdx.x * per + min((int)blockIdx.x, extra);
    const int o1 = o0 + per + ((int)blockIdx.x < extra ? 1 : 0);
    if (o0 >= o1) return;   // nothing issued yet

    const uint32_t ring = smem_addr(rowt_ring);
    const uint32_t bars = ring + (uint32_t)(g.NS * g.stage);
    volatile int *abort_flag =
        reinterpret_cast<volatile int *>(rowt_ring + g.NS * g.stage + 8 * g.NS);

    // Producer (thread 0 only): input rows in consumption order.
    RowTRun prun{};
    int pnext_u = 0, pj = 0;
    int pissued = 0, preleased = 0;
    bool pdone = false;
    auto issue = [&]() {
        if (pdone) return;
        const int slot = pissued & (g.NS - 1);
        const uint32_t bar = bars + 8u * (uint32_t)slot;
        mbar_arrive_expect_tx(bar, (uint32_t)g.box_bytes);
        tma_load_4d(ring + (uint32_t)(slot * g.stage), &xmap, bar, prun.hc * g.CVc * VEC,
                    ((prun.cc * g.OWc - g.sh0 + p.pbw) >> 1) - KE / 2, prun.j0 + pj, prun.n);
        ++pissued;
        if (++pj == prun.nj) {
            if (pnext_u >= o1) {
                pdone = true;
            } else {
                prun = rowt_run_at(pnext_u, o1, p, g, K);
                pnext_u += prun.rows;
                pj = 0;
            }
        }
    };

    if (t == 0) {
        tma_prefetch_map(&xmap);
        for (int i = 0; i < g.NS; ++i) mbar_init(bars + 8u * i, 1);
        *abort_flag = 0;
        fence_barrier_init();
        prun = rowt_run_at(o0, o1, p, g, K);
        pnext_u = o0 + prun.rows;
        for (int i = 0; i < g.NS; ++i) issue();
    }
    __syncthreads();

    float2 wr[K][K][P];
    float2 bias[P];
    int loaded_hc = -1;
    int cnext = 0;       // next sequence number to wait for
    int cseen = 0;       // boxes seen to arrive
    int cbase = 0;       // sequence number of the current run's first input row
    bool bad = false;
    const uint32_t win_off = (uint32_t)(cvl * VB + pg * (S / 2) * g.pitch);
    int u = o0;
    while (u < o1) {
        const RowTRun run = rowt_run_at(u, o1, p, g, K);
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
                        const T *wp = w + (int64_t)(c0 + 2 * k) * p.ws[0] + kh * p.ws[2] + kw * p.ws[3];
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
        const int iw0 = run.cc * g.OWc - g.sh0 + pg * S;
        T *yn = y + (int64_t)run.n * p.ys[0] + (active ? c0 : 0);
        const int oh_end = run.oh0 + run.rows;
        const bool cols_full = iw0 >= 0 && iw0 + S <= p.OW;   // no column check needed
        // Output rows in pairs (r, r + 1) with r + pad even: row r takes the
        // even taps kh = 2a and row r + 1 the odd taps kh = 2a + 1, both from
        // input row m - a (m = (r + pad)/2), so each input row's window is
        // loaded once for the pair.  A pair may stick out of the run by one
        // row at either end; that row is not stored.
        for (int r = run.oh0 - ((run.oh0 + p.pbh) & 1); r < oh_end; r += 2) {
            const int m = (r + p.pbh) >> 1;
            const int need = cbase + (m - run.j0) + 1;
            while (cnext < need) {
                if (!bad) {
                    if (mbar_wait(bars + 8u * (uint32_t)(cnext & (g.NS - 1)),
                                  (uint32_t)((cnext >> g.ns_log2) & 1), abort_flag)) {
                        ++cseen;
                    } else {
                        bad = true;
                        *abort_flag = 1;
                    }
                }
                ++cnext;
            }
            if (t == 0 && *abort_flag) pdone = true;
            float2 acc[2][S][P];
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < S; ++i)
#pragma unroll
                    for (int k = 0; k < P; ++k) acc[h][i][k] = bias[k];
#pragma unroll
            for (int a = 0; a <= KE / 2; ++a) {
                const int seq = cbase + (m - a - run.j0);
                const uint32_t st = ring + (uint32_t)((seq & (g.NS - 1)) * g.stage) + win_off;
                float2 xr[WIN][P];
#pragma unroll
                for (int q = 0; q < WIN; ++q) {
                    V v;
                    Lds<VB>::load(v, st + (uint32_t)(q * g.pitch));
                    widen<T, VEC>(v, xr[q]);
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int kh = 2 * a + h;
                    if (kh >= K) continue;   // compile time
#pragma unroll
                    for (int i = 0; i < S; ++i)
#pragma unroll
                        for (int kw = 0; kw < K; ++kw) {
                            if (((i - kw) & 1) != 0) continue;   // compile time
#pragma unroll
                            for (int k = 0; k < P; ++k)
                                fma2_packed(acc[h][i][k], wr[kh][kw][k], xr[(i - kw + KE) / 2][k]);
                        }
                }
            }
            if (bad)
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int i = 0; i < S; ++i)
#pragma unroll
                        for (int k = 0; k < P; ++k) acc[h][i][k] = make_float2(kNaN, kNaN);
            if (active) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int oh = r + h;
                    if (oh < run.oh0 || oh >= oh_end) continue;
                    T *yrow = yn + (int64_t)oh * p.ys[2] + (int64_t)iw0 * p.ys[3];
                    if (cols_full) {
#pragma unroll
                        for (int i = 0; i < S; ++i)
                            IO::store(yrow + i * p.ys[3], pack_pairs<T, VEC>(acc[h][i]));
                    } else {
#pragma unroll
                        for (int i = 0; i < S; ++i) {
                            const int iw = iw0 + i;
                            if (iw >= 0 && iw < p.OW)
                                IO::store(yrow + i * p.ys[3], pack_pairs<T, VEC>(acc[h][i]));
                        }
                    }
                }
            }
            __syncthreads();   // every thread is done with the rows it read
            if (t == 0) {
                // Input rows below the first one the next pair reads are
                // free (all of the run's after its last pair).
                int rel = cbase + run.nj;
                if (r + 2 < oh_end) {
                    const int q = m + 1 - KE / 2 - run.j0;
                    rel = cbase + (q > 0 ? q : 0);
                }
                if (rel > preleased) preleased = rel;
                while (!pdone && pissued < preleased + g.NS) issue();
            }
        }
        cbase += run.nj;
    }
    // After a failed wait, boxes issued but never seen to arrive may still be
    // landing in this CTA's shared memory: wait for each once more (bounded).
    if (t == 0 && *abort_flag)
        for (int q = cseen; q < pissued; ++q)
            (void)mbar_wait(bars + 8u * (uint32_t)(q & (g.NS - 1)), (uint32_t)((q >> g.ns_log2) & 1));
}

template <typename T, int K>
cudaError_t row8t_launch_t(const Params &p, const Ptrs &q, cudaStream_t s) {
    constexpr int VEC = row8_vec<T>(K);
    RowTGeom g;
    if (!rowt_geometry<T, K>(p, g)) return cudaErrorNotSupported;
    const uint64_t es = sizeof(T);
    const uint64_t dims[4] = {(uint64_t)p.C_in, (uint64_t)p.W, (uint64_t)p.H, (uint64_t)p.N};
    const uint64_t strides[3] = {(uint64_t)p.xs[3] * es, (uint64_t)p.xs[2] * es,
                                 (uint64_t)p.xs[0] * es};
    const uint32_t box[4] = {(uint32_t)(g.CVc * VEC), (uint32_t)g.Wq, 1u, 1u};
    CUtensorMap map;
    if (!tma_encode_4d(&map, tma_dtype<T>(), q.x, dims, strides, box)) return cudaErrorInvalidValue;
    const size_t smem = (size_t)g.NS * g.stage + 8 * (size_t)g.NS + 16;
    cudaError_t e = cudaFuncSetAttribute(row8t_kernel<T, K>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_kernel(row8t_kernel<T, K>, dim3(g.ctas), dim3(g.CVc * g.PG), smem, s, map,
                   static_cast<const T *>(q.w), static_cast<const T *>(q.b),
                   static_cast<T *>(q.y), p, g);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename T>
cudaError_t row8t_launch_dtype(const Params &p, const Ptrs &q, cudaStream_t s) {
    switch (p.KH) {
    case 3: return row8t_launch_t<T, 3>(p, q, s);
    case 5: return row8t_launch_t<T, 5>(p, q, s);
    case 7: return row8t_launch_t<T, 7>(p, q, s);
    }
    return cudaErrorNotSupported;
}

template <typename T>
bool row8t_fits_dtype(const Params &p) {
    RowTGeom g;
    switch (p.KH) {
    case 3: return rowt_geometry<T, 3>(p, g);
    case 5: return rowt_geometry<T, 5>(p, g);
    case 7: return rowt_geometry<T, 7>(p, g);
    }
    return false;
}

cudaError_t row8t_launch_f32(const Params &p, const Ptrs &q, cudaStream_t s);
cudaError_t row8t_launch_f16(const Params &p, const Ptrs &q, cudaStream_t s);
cudaError_t row8t_launch_bf16(const Params &p, const Ptrs &q, cudaStream_t s);

}  // namespace gconv
