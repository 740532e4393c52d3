/*
 * conv_oracle.c -- TEST INFRASTRUCTURE, not part of the product path.
 *
 * A plain, slow, obviously correct CPU fp64 reference for 2-D grouped and
 * depthwise convolution.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may call it.  It shares no code, header or constant with
 * the CUDA library.
 *
 * What it computes (cross-correlation, no kernel flip, zero padding):
 *
 *   y[n, co, oh, ow] = b[co]
 *       + sum_{ci < Cin_g, kh < KH, kw < KW, (ih, iw) inside the input}
 *             w[co, ci, kh, kw] * x[n, g*Cin_g + ci, ih, iw]
 *   with g = co / Cout_g, ih = oh*sh - pbh + kh, iw = ow*sw - pbw + kw.
 *
 * Sources:
 *  - tap indexing: torch/_inductor/kernel/conv.py, LOOP_BODY_2D (the input
 *    row is the tap index minus the padding plus the output row times the
 *    stride; taps outside [0, IN_H) x [0, IN_W) are masked to zero);
 *  - channel-to-group mapping: torch/_inductor/kernel/conv.py,
 *    conv2d_template (group g reads input channels [g*GROUP_IN_C, ...) and
 *    writes output channels [g*GROUP_OUT_C, ...));
 *  - separate padding before and after each spatial dim: executorch PR
 *    #25084 "Add triton::convolution and the conv routing framework",
 *    description, second paragraph (explicit padding_before/padding_after);
 *  - fp64 as the reference precision: executorch PR #25085 "Route 2-D
 *    depthwise and few-channel grouped convolutions to a Triton
 *    direct-stencil kernel", description, last paragraph (schedules are
 *    tested against an FP64 reference).
 *
 * Alongside y it returns bound[n, co, oh, ow] = sum over the same taps of
 * |w * x| plus |b[co]|, the scale of the parity tolerance.  The bias counts
 * as one more product term (b times a constant input of 1): with it left
 * out, an output dominated by the bias could not meet the tolerance even
 * when it is the exact value correctly rounded to fp16 or bf16.
 *
 * Output spatial size: the number of window starts t = 0, s, 2s, ... in the
 * explicitly padded input (length H + pb + pa) with t + K <= H + pb + pa,
 * i.e. floor((H + pb + pa - K) / s) + 1 when H + pb + pa >= K, else none.
 *
 * All arrays are dense and in logical order: x [N, C_in, H, W],
 * w [C_out, Cin_g, KH, KW], b [C_out] (or NULL), y and bound
 * [N, C_out, OH, OW].  Built with -ffp-contract=off so products and sums
 * are rounded separately on every host.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Number of window starts along one spatial dim; -1 if the window does not
 * fit even once or an argument is out of range. */
int64_t oracle_out_size(int64_t in, int64_t k, int64_t s, int64_t pb, int64_t pa)
{
    if (in < 0 || k < 1 || s < 1 || pb < 0 || pa < 0) return -1;
    int64_t padded = in + pb + pa;
    if (padded < k) return -1;
    int64_t count = 0;
    for (int64_t t = 0; t + k <= padded; t += s) ++count;
    return count;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* One output element: the sum over the group's input channels and the taps. */
static void one_output(const double *x, const double *w, const double *b,
                       int64_t C_in, int64_t H, int64_t W,
                       int64_t Cin_g, int64_t Cout_g, int64_t KH, int64_t KW,
                       int64_t sh, int64_t sw, int64_t pbh, int64_t pbw,
                       int64_t n, int64_t co, int64_t oh, int64_t ow,
                       double *y_out, double *bound_out)
{
    int64_t g = co / Cout_g;
    double acc = 0.0, sabs = 0.0;
    for (int64_t ci = 0; ci < Cin_g; ++ci) {
        int64_t c = g * Cin_g + ci;
        for (int64_t kh = 0; kh < KH; ++kh) {
            int64_t ih = oh * sh - pbh + kh;
            if (ih < 0 || ih >= H) continue;
            for (int64_t kw = 0; kw < KW; ++kw) {
                int64_t iw = ow * sw - pbw + kw;
                if (iw < 0 || iw >= W) continue;
                double xv = x[((n * C_in + c) * H + ih) * W + iw];
                double wv = w[((co * Cin_g + ci) * KH + kh) * KW + kw];
                double p = wv * xv;
                acc += p;
                sabs += fabs(p);
            }
        }
    }
    if (b) {
        acc += b[co];
        sabs += fabs(b[co]);
    }
    *y_out = acc;
    *bound_out = sabs;
}

static int check_args(int64_t N, int64_t C_in, int64_t H, int64_t W,
                      int64_t C_out, int64_t groups, int64_t KH, int64_t KW,
                      int64_t sh, int64_t sw, int64_t pbh, int64_t pbw,
                      int64_t pah, int64_t paw, int64_t *OH, int64_t *OW)
{
    if (N < 0 || C_in < 0 || C_out < 0 || groups < 1) return 1;
    if (C_in % groups != 0 || C_out % groups != 0) return 1;
    *OH = oracle_out_size(H, KH, sh, pbh, pah);
    *OW = oracle_out_size(W, KW, sw, pbw, paw);
    if (*OH < 0 || *OW < 0) return 1;
    return 0;
}

/* Full convolution.  Returns 0 on success, 1 on bad arguments. */
int oracle_conv2d_f64(const double *x, const double *w, const double *b,
                      int64_t N, int64_t C_in, int64_t H, int64_t W,
                      int64_t C_out, int64_t groups, int64_t KH, int64_t KW,
                      int64_t sh, int64_t sw, int64_t pbh, int64_t pbw,
                      int64_t pah, int64_t paw, double *y, double *bound)
{
    int64_t OH, OW;
    if (check_args(N, C_in, H, W, C_out, groups, KH, KW, sh, sw, pbh, pbw,
                   pah, paw, &OH, &OW))
        return 1;
    const int64_t Cin_g = C_in / groups, Cout_g = C_out / groups;
    const int64_t planes = N * C_out;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t p = 0; p < planes; ++p) {
        int64_t n = p / C_out, co = p % C_out;
        for (int64_t oh = 0; oh < OH; ++oh)
            for (int64_t ow = 0; ow < OW; ++ow) {
                int64_t o = ((n * C_out + co) * OH + oh) * OW + ow;
                one_output(x, w, b, C_in, H, W, Cin_g, Cout_g, KH, KW, sh, sw,
                           pbh, pbw, n, co, oh, ow, &y[o], &bound[o]);
            }
    }
    return 0;
}

/* Selected outputs only: pts holds npts rows of (n, co, oh, ow). */
int oracle_conv2d_f64_points(const double *x, const double *w, const double *b,
                             int64_t N, int64_t C_in, int64_t H, int64_t W,
                             int64_t C_out, int64_t groups, int64_t KH, int64_t KW,
                             int64_t sh, int64_t sw, int64_t pbh, int64_t pbw,
                             int64_t pah, int64_t paw, int64_t npts,
                             const int64_t *pts, double *y, double *bound)
{
    int64_t OH, OW;
    if (check_args(N, C_in, H, W, C_out, groups, KH, KW, sh, sw, pbh, pbw,
                   pah, paw, &OH, &OW))
        return 1;
    for (int64_t i = 0; i < npts; ++i) {
        const int64_t *q = pts + 4 * i;
        if (q[0] < 0 || q[0] >= N || q[1] < 0 || q[1] >= C_out || q[2] < 0 ||
            q[2] >= OH || q[3] < 0 || q[3] >= OW)
            return 1;
    }
    const int64_t Cin_g = C_in / groups, Cout_g = C_out / groups;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < npts; ++i) {
        const int64_t *q = pts + 4 * i;
        one_output(x, w, b, C_in, H, W, Cin_g, Cout_g, KH, KW, sh, sw, pbh,
                   pbw, q[0], q[1], q[2], q[3], &y[i], &bound[i]);
    }
    return 0;
}
