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
 *   with g = co / Cout_g, ih = oh*sh - pbh + kh*dh, iw = ow*sw - pbw + kw*dw
 *   (dh, dw: dilation, the spacing of the taps; 1 for the direct stencil).
 *
 * Also here, each from its own definition (no shared arithmetic with the
 * forward beyond the index rules they state):
 *  - the transposed convolution (executorch PR #25091 "Run transposed
 *    convolutions on the implicit-GEMM template", description, second
 *    paragraph): output o reads, at tap k, input (o + pad_before - k*d) / s
 *    when that is an integer inside the input, and the weight is
 *    [C_in, C_out / groups, KH, KW] (its first two dims swapped relative to
 *    the forward weight);
 *  - the gradients of the forward convolution with respect to x, w and b
 *    (the backward that torch/_inductor/kernel/conv.py,
 *    convolution_backward_lowering, lowers: grad_input, grad_weight and
 *    grad_bias = the sum of grad_output over batch and space), written as
 *    the derivative of the forward sum term by term: every product
 *    w * x that the forward adds into y[n, co, oh, ow] sends
 *    gy[n, co, oh, ow] * w to dx at x's index and gy[n, co, oh, ow] * x to dw
 *    at w's index.
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
 * |w * x| (the bias is not a term of it), the scale of the parity
 * tolerance tol * sum|w * x| + 1e-6.
 *
 * Output spatial size: the number of window starts t = 0, s, 2s, ... in the
 * explicitly padded input (length H + pb + pa) with t + E <= H + pb + pa,
 * E = d*(K-1)+1 the window's span, i.e. floor((H + pb + pa - E) / s) + 1
 * when H + pb + pa >= E, else none.
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
 * fit even once or an argument is out of range.  A window of k taps spaced
 * d apart spans d*(k-1)+1 input positions. */
int64_t oracle_out_size(int64_t in, int64_t k, int64_t s, int64_t pb, int64_t pa,
                        int64_t d)
{
    if (in < 0 || k < 1 || s < 1 || d < 1 || pb < 0 || pa < 0) return -1;
    int64_t padded = in + pb + pa;
    int64_t span = d * (k - 1) + 1;
    if (padded < span) return -1;
    int64_t count = 0;
    for (int64_t t = 0; t + span <= padded; t += s) ++count;
    return count;
}

/* Output length of a transposed convolution along one dim: every input
 * position i places its k taps at i*s + j*d (j < k), so the uncropped output
 * spans (in-1)*s + d*(k-1) + 1 positions; output_padding op adds op more at
 * the end, then pb positions are cropped before and pa after.  -1 when an
 * argument is out of range or nothing is left. */
int64_t oracle_transposed_out_size(int64_t in, int64_t k, int64_t s, int64_t pb,
                                   int64_t pa, int64_t op, int64_t d)
{
    if (in < 1 || k < 1 || s < 1 || d < 1 || pb < 0 || pa < 0 || op < 0) return -1;
    int64_t full = 0;
    /* the last position any tap reaches, plus one */
    for (int64_t i = 0; i < in; ++i)
        for (int64_t j = 0; j < k; ++j)
            if (i * s + j * d + 1 > full) full = i * s + j * d + 1;
    int64_t out = full + op - pb - pa;
    return out >= 1 ? out : -1;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for the later calls (a timing aid; the results do not depend on it). */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* One output element: the sum over the group's input channels and the taps. */
static void one_output(const double *x, const double *w, const double *b,
                       int64_t C_in, int64_t H, int64_t W,
                       int64_t Cin_g, int64_t Cout_g, int64_t KH, int64_t KW,
                       int64_t sh, int64_t sw, int64_t pbh, int64_t pbw,
                       int64_t dh, int64_t dw,
                       int64_t n, int64_t co, int64_t oh, int64_t ow,
                       double *y_out, double *bound_out)
{
    int64_t g = co / Cout_g;
    double acc = 0.0, sabs = 0.0;
    for (int64_t ci = 0; ci < Cin_g; ++ci) {
        int64_t c = g * Cin_g + ci;
        for (int64_t kh = 0; kh < KH; ++kh) {
            int64_t ih = oh * sh - pbh + kh * dh;
            if (ih < 0 || ih >= H) continue;
            for (int64_t kw = 0; kw < KW; ++kw) {
                int64_t iw = ow * sw - pbw + kw * dw;
                if (iw < 0 || iw >= W) continue;
                double xv = x[((n * C_in + c) * H + ih) * W + iw];
                double wv = w[((co * Cin_g + ci) * KH + kh) * KW + kw];
                double p = wv * xv;
                acc += p;
                sabs += fabs(p);
            }
        }
    }
    if (b) acc += b[co];
    *y_out = acc;
    *bound_out = sabs;
}

static int check_args(int64_t N, int64_t C_in, int64_t H, int64_t W,
                      int64_t C_out, int64_t groups, int64_t KH, int64_t KW,
                      int64_t sh, int64_t sw, int64_t pbh, int64_t pbw,
                      int64_t pah, int64_t paw, int64_t dh, int64_t dw,
                      int64_t *OH, int64_t *OW)
{
    if (N < 0 || C_in < 0 || C_out < 0 || groups < 1) return 1;
    if (C_in % groups != 0 || C_out % groups != 0) return 1;
    *OH = oracle_out_size(H, KH, sh, pbh, pah, dh);
    *OW = oracle_out_size(W, KW, sw, pbw, paw, dw);
    if (*OH < 0 || *OW < 0) return 1;
    return 0;
}

/* Full convolution.  Returns 0 on success, 1 on bad arguments. */
int oracle_conv2d_f64(const double *x, const double *w, const double *b,
                      int64_t N, int64_t C_in, int64_t H, int64_t W,
                      int64_t C_out, int64_t groups, int64_t KH, int64_t KW,
                      int64_t sh, int64_t sw, int64_t pbh, int64_t pbw,
                      int64_t pah, int64_t paw, int64_t dh, int64_t dw,
                      double *y, double *bound)
{
    int64_t OH, OW;
    if (check_args(N, C_in, H, W, C_out, groups, KH, KW, sh, sw, pbh, pbw,
                   pah, paw, dh, dw, &OH, &OW))
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
                           pbh, pbw, dh, dw, n, co, oh, ow, &y[o], &bound[o]);
            }
    }
    return 0;
}

/* Selected outputs only: pts holds npts rows of (n, co, oh, ow). */
int oracle_conv2d_f64_points(const double *x, const double *w, const double *b,
                             int64_t N, int64_t C_in, int64_t H, int64_t W,
                             int64_t C_out, int64_t groups, int64_t KH, int64_t KW,
                             int64_t sh, int64_t sw, int64_t pbh, int64_t pbw,
                             int64_t pah, int64_t paw, int64_t dh, int64_t dw,
                             int64_t npts, const int64_t *pts, double *y,
                             double *bound)
{
    int64_t OH, OW;
    if (check_args(N, C_in, H, W, C_out, groups, KH, KW, sh, sw, pbh, pbw,
                   pah, paw, dh, dw, &OH, &OW))
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
                   pbw, dh, dw, q[0], q[1], q[2], q[3], &y[i], &bound[i]);
    }
    return 0;
}

/* ------------------------------------------------------------ transposed */

/* One output of the transposed convolution: a gather over the group's
 * input channels and the taps whose input index is a whole number inside
 * the input.  w is [C_in, Cout_g, KH, KW]. */
static void one_transposed(const double *x, const double *w, const double *b,
                           int64_t C_in, int64_t H, int64_t W,
                           int64_t Cin_g, int64_t Cout_g, int64_t KH, int64_t KW,
                           int64_t sh, int64_t sw, int64_t pbh, int64_t pbw,
                           int64_t dh, int64_t dw,
                           int64_t n, int64_t co, int64_t oh, int64_t ow,
                           double *y_out, double *bound_out)
{
    int64_t g = co / Cout_g, j = co - g * Cout_g;
    double acc = 0.0, sabs = 0.0;
    for (int64_t ci = 0; ci < Cin_g; ++ci) {
        int64_t c = g * Cin_g + ci;
        for (int64_t kh = 0; kh < KH; ++kh) {
            int64_t th = oh + pbh - kh * dh;          /* = ih * sh when it lands */
            if (th < 0 || th % sh != 0) continue;
            int64_t ih = th / sh;
            if (ih >= H) continue;
            for (int64_t kw = 0; kw < KW; ++kw) {
                int64_t tw = ow + pbw - kw * dw;
                if (tw < 0 || tw % sw != 0) continue;
                int64_t iw = tw / sw;
                if (iw >= W) continue;
                double xv = x[((n * C_in + c) * H + ih) * W + iw];
                double wv = w[((c * Cout_g + j) * KH + kh) * KW + kw];
                double p = wv * xv;
                acc += p;
                sabs += fabs(p);
            }
        }
    }
    if (b) acc += b[co];
    *y_out = acc;
    *bound_out = sabs;
}

static int check_transposed(int64_t N, int64_t C_in, int64_t H, int64_t W,
                            int64_t C_out, int64_t groups, int64_t KH, int64_t KW,
                            int64_t sh, int64_t sw, int64_t pbh, int64_t pbw,
                            int64_t pah, int64_t paw, int64_t oph, int64_t opw,
                            int64_t dh, int64_t dw, int64_t *OH, int64_t *OW)
{
    if (N < 0 || C_in < 0 || C_out < 0 || groups < 1) return 1;
    if (C_in % groups != 0 || C_out % groups != 0) return 1;
    *OH = oracle_transposed_out_size(H, KH, sh, pbh, pah, oph, dh);
    *OW = oracle_transposed_out_size(W, KW, sw, pbw, paw, opw, dw);
    if (*OH < 0 || *OW < 0) return 1;
    return 0;
}

/* Full transposed convolution: x [N, C_in, H, W], w [C_in, C_out/groups, KH,
 * KW], b [C_out] or NULL, y and bound [N, C_out, OH, OW].  0 on success. */
int oracle_conv_transpose2d_f64(const double *x, const double *w, const double *b,
                                int64_t N, int64_t C_in, int64_t H, int64_t W,
                                int64_t C_out, int64_t groups, int64_t KH, int64_t KW,
                                int64_t sh, int64_t sw, int64_t pbh, int64_t pbw,
                                int64_t pah, int64_t paw, int64_t oph, int64_t opw,
                                int64_t dh, int64_t dw, double *y, double *bound)
{
    int64_t OH, OW;
    if (check_transposed(N, C_in, H, W, C_out, groups, KH, KW, sh, sw, pbh, pbw,
                         pah, paw, oph, opw, dh, dw, &OH, &OW))
        return 1;
    const int64_t Cin_g = C_in / groups, Cout_g = C_out / groups;
    const int64_t planes = N * C_out;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t p = 0; p < planes; ++p) {
        int64_t n = p / C_out, co = p % C_out;
        for (int64_t oh = 0; oh < OH; ++oh)
            for (int64_t ow = 0; ow < OW; ++ow) {
                int64_t o = ((n * C_out + co) * OH + oh) * OW + ow;
                one_transposed(x, w, b, C_in, H, W, Cin_g, Cout_g, KH, KW, sh, sw,
                               pbh, pbw, dh, dw, n, co, oh, ow, &y[o], &bound[o]);
            }
    }
    return 0;
}

/* Selected outputs of the transposed convolution (pts: npts rows of
 * (n, co, oh, ow)). */
int oracle_conv_transpose2d_f64_points(const double *x, const double *w, const double *b,
                                       int64_t N, int64_t C_in, int64_t H, int64_t W,
                                       int64_t C_out, int64_t groups, int64_t KH,
                                       int64_t KW, int64_t sh, int64_t sw, int64_t pbh,
                                       int64_t pbw, int64_t pah, int64_t paw,
                                       int64_t oph, int64_t opw, int64_t dh, int64_t dw,
                                       int64_t npts, const int64_t *pts, double *y,
                                       double *bound)
{
    int64_t OH, OW;
    if (check_transposed(N, C_in, H, W, C_out, groups, KH, KW, sh, sw, pbh, pbw,
                         pah, paw, oph, opw, dh, dw, &OH, &OW))
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
        one_transposed(x, w, b, C_in, H, W, Cin_g, Cout_g, KH, KW, sh, sw, pbh,
                       pbw, dh, dw, q[0], q[1], q[2], q[3], &y[i], &bound[i]);
    }
    return 0;
}

/* --------------------------------------------------------------- backward */

/* Gradients of the forward convolution (same geometry arguments as
 * oracle_conv2d_f64) given gy [N, C_out, OH, OW]:
 *   dx [N, C_in, H, W]:          every forward product w * x sends gy * w to
 *                                dx at x's index;
 *   dw [C_out, Cin_g, KH, KW]:   ... and gy * x to dw at w's index;
 *   db [C_out]:                  the sum of gy over n, oh, ow.
 * Each *_bound array receives the sum of the absolute values of the same
 * terms (the parity tolerance scale).  Any of the outputs may be NULL (with
 * its bound) to skip it.  dx is scattered one image at a time (images in
 * parallel: their dx slices are disjoint); dw and db one output channel at a
 * time (channels in parallel).  0 on success. */
int oracle_conv2d_backward_f64(const double *x, const double *w, const double *gy,
                               int64_t N, int64_t C_in, int64_t H, int64_t W,
                               int64_t C_out, int64_t groups, int64_t KH, int64_t KW,
                               int64_t sh, int64_t sw, int64_t pbh, int64_t pbw,
                               int64_t pah, int64_t paw, int64_t dh, int64_t dw,
                               double *dx, double *dx_bound, double *dwt,
                               double *dw_bound, double *db, double *db_bound)
{
    int64_t OH, OW;
    if (check_args(N, C_in, H, W, C_out, groups, KH, KW, sh, sw, pbh, pbw,
                   pah, paw, dh, dw, &OH, &OW))
        return 1;
    const int64_t Cin_g = C_in / groups, Cout_g = C_out / groups;
    if (dx) {
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t n = 0; n < N; ++n) {
            for (int64_t i = 0; i < C_in * H * W; ++i) {
                dx[n * C_in * H * W + i] = 0.0;
                dx_bound[n * C_in * H * W + i] = 0.0;
            }
            for (int64_t co = 0; co < C_out; ++co) {
                int64_t g = co / Cout_g;
                for (int64_t oh = 0; oh < OH; ++oh)
                    for (int64_t ow = 0; ow < OW; ++ow) {
                        double gv = gy[((n * C_out + co) * OH + oh) * OW + ow];
                        for (int64_t ci = 0; ci < Cin_g; ++ci) {
                            int64_t c = g * Cin_g + ci;
                            for (int64_t kh = 0; kh < KH; ++kh) {
                                int64_t ih = oh * sh - pbh + kh * dh;
                                if (ih < 0 || ih >= H) continue;
                                for (int64_t kw = 0; kw < KW; ++kw) {
                                    int64_t iw = ow * sw - pbw + kw * dw;
                                    if (iw < 0 || iw >= W) continue;
                                    double p = gv * w[((co * Cin_g + ci) * KH + kh) * KW + kw];
                                    int64_t xi = ((n * C_in + c) * H + ih) * W + iw;
                                    dx[xi] += p;
                                    dx_bound[xi] += fabs(p);
                                }
                            }
                        }
                    }
            }
        }
    }
    if (dwt || db) {
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t co = 0; co < C_out; ++co) {
            int64_t g = co / Cout_g;
            double bsum = 0.0, babs = 0.0;
            if (dwt)
                for (int64_t i = 0; i < Cin_g * KH * KW; ++i) {
                    dwt[co * Cin_g * KH * KW + i] = 0.0;
                    dw_bound[co * Cin_g * KH * KW + i] = 0.0;
                }
            for (int64_t n = 0; n < N; ++n)
                for (int64_t oh = 0; oh < OH; ++oh)
                    for (int64_t ow = 0; ow < OW; ++ow) {
                        double gv = gy[((n * C_out + co) * OH + oh) * OW + ow];
                        bsum += gv;
                        babs += fabs(gv);
                        if (!dwt) continue;
                        for (int64_t ci = 0; ci < Cin_g; ++ci) {
                            int64_t c = g * Cin_g + ci;
                            for (int64_t kh = 0; kh < KH; ++kh) {
                                int64_t ih = oh * sh - pbh + kh * dh;
                                if (ih < 0 || ih >= H) continue;
                                for (int64_t kw = 0; kw < KW; ++kw) {
                                    int64_t iw = ow * sw - pbw + kw * dw;
                                    if (iw < 0 || iw >= W) continue;
                                    double p = gv * x[((n * C_in + c) * H + ih) * W + iw];
                                    int64_t wi = ((co * Cin_g + ci) * KH + kh) * KW + kw;
                                    dwt[wi] += p;
                                    dw_bound[wi] += fabs(p);
                                }
                            }
                        }
                    }
            if (db) {
                db[co] = bsum;
                db_bound[co] = babs;
            }
        }
    }
    return 0;
}
