/*
 * gconv.h -- C ABI of the GB300 direct-stencil convolution library.
 *
 * The operation: 2-D depthwise and few-channel grouped convolution
 * (cross-correlation, zero padding) with
 *   - groups of 1..8 input channels and any number of output channels each
 *     (any depthwise channel multiplier),
 *   - kernels from 1x1 to 9x9 (KH and KW independent), any stride >= 1,
 *   - explicit, possibly asymmetric, padding before and after each spatial dim,
 *   - fp32, fp16 or bf16 tensors (all of one dtype), fp32 accumulation and a
 *     single round-to-nearest-even cast of (sum + bias) at the end,
 *   - NCHW- or channels-last-ordered input, optional bias.
 * The envelope is the one of the direct-stencil template in executorch PR
 * #25085 "Route 2-D depthwise and few-channel grouped convolutions to a
 * Triton direct-stencil kernel" (description, second paragraph), which takes
 * dilation 1 only.  Around it the same library offers, on the same
 * kernels' designs:
 *   - dilation >= 1 (taps d apart) and 1-D convolutions (the height-1 case,
 *     conv1d_bind), the calls executorch PR #25084 says Inductor's templates
 *     cannot compile (description, first paragraph);
 *   - the transposed convolution of executorch PR #25091 "Run transposed
 *     convolutions on the implicit-GEMM template" (description, second
 *     paragraph; conv_transpose_bind, conv_transpose_forward);
 *   - the backward of the forward convolution (the gradients that
 *     torch/_inductor/kernel/conv.py, convolution_backward_lowering,
 *     lowers: conv_backward_input, conv_backward_weight).
 *
 * Semantics.  For output (n, co, oh, ow), with g = co / Cout_g:
 *   y = b[co] + sum_{ci, kh, kw} w[co, ci, kh, kw] * x[n, g*Cin_g + ci, ih, iw],
 *   ih = oh*stride_h - pad_before_h + kh*dil_h,
 *   iw = ow*stride_w - pad_before_w + kw*dil_w,
 * where taps with (ih, iw) outside the input contribute zero.  The tap
 * indexing is the one of torch/_inductor/kernel/conv.py, LOOP_BODY_2D; the
 * channel-to-group mapping that of conv2d_template in the same file; the
 * explicit padding_before / padding_after pair that of the canonical
 * convolution op in executorch PR #25084 "Add triton::convolution and the conv
 * routing framework" (description, second paragraph).
 *
 * Call sequence (PR #25084, second paragraph: the arguments are bound and
 * validated once, the output layout is computed by one function, the output
 * is allocated once by the caller and the kernels only write into it):
 *   conv_bind -> out_shape_and_stride -> caller allocates y ->
 *   conv_dw_forward (Cin_g == 1) or conv_grouped_forward (1 <= Cin_g <= 8).
 * Transposed: conv_transpose_bind -> out_shape_and_stride -> allocate y ->
 *   conv_transpose_forward.
 * Backward of a forward desc: grad_input_shape_and_stride -> allocate dx ->
 *   conv_backward_input; conv_backward_weight_workspace_size -> allocate
 *   the workspace, dw and db -> conv_backward_weight.
 *
 * Ownership.  The caller owns every buffer, including the one workspace the
 * library asks for (conv_backward_weight's).  The library allocates no
 * memory, keeps no pointer after a call returns and never synchronises;
 * kernels run asynchronously on the caller's stream.
 *
 * Ordering.  Each forward is one kernel launched with programmatic
 * dependent launch: it may start while the previous kernel on the stream is
 * finishing, but it waits for that kernel's memory before its first read of
 * x, w or bias, so stream order is kept exactly (a forward may consume the
 * previous kernel's output).  It also lets the next kernel on the stream
 * start early; a next kernel that does not opt in to programmatic launch
 * simply waits for it to complete, as usual.
 *
 * Errors.  Every entry point returns a gconv_status; nothing throws or
 * aborts across the ABI.  conv_strerror() names a status.
 *
 * Threads.  All entry points are re-entrant.  The process-wide schedule
 * override (conv_force_schedule) and the injected-error hook are atomics.
 */
#ifndef GCONV_H
#define GCONV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (the same object as cudaStream_t / CUstream).
 * NULL means the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st *gconv_stream;

typedef enum gconv_dtype {
    GCONV_F32 = 0,
    GCONV_F16 = 1,
    GCONV_BF16 = 2
} gconv_dtype;

typedef enum gconv_status {
    GCONV_OK = 0,
    GCONV_ERR_NULL = 1,          /* a required pointer is NULL, or bias presence mismatches */
    GCONV_ERR_RANK = 2,          /* x not rank 3/4, w not rank 4, bias not rank 1 */
    GCONV_ERR_DTYPE = 3,         /* unknown dtype code */
    GCONV_ERR_SHAPE = 4,         /* channel/group/weight/bias size mismatch, stride < 1, negative size */
    GCONV_ERR_UNSUPPORTED = 5,   /* dilation < 1, KH or KW outside [1, 9], Cin_g > 8,
                                    Cin_g != 1 on conv_dw_forward */
    GCONV_ERR_PADDING = 6,       /* negative padding, or the window never fits the padded input */
    GCONV_ERR_ALIGN = 7,         /* a forced schedule needs alignment the pointers lack */
    GCONV_ERR_CUDA = 8,          /* a CUDA launch failed (cudaGetLastError after the launch) */
    GCONV_ERR_INTERNAL = 9,      /* descriptor not produced by conv_bind, or a size overflow */
    GCONV_ERR_LAYOUT = 10,       /* x is neither NCHW- nor channels-last-ordered */
    GCONV_ERR_SCHEDULE = 11,     /* a forced schedule does not support this call */
    GCONV_ERR_KIND = 12,         /* desc of another operation (forward vs transposed) */
    GCONV_ERR_WORKSPACE = 13,    /* workspace missing, too small or misaligned */
    GCONV_ERR_SCRATCH_LIMIT = 14 /* conv_backward_weight_noalloc: the problem needs more
                                    scratch than its fixed device buffer holds */
} gconv_status;

/* The five schedules of the direct-stencil template (PR #25085, second
 * paragraph), re-designed for sm_103a, plus: a tensor-core schedule for
 * 4- and 8-channel groups; a channels-last depthwise schedule for the
 * shapes outside the others' reach (dilated, 1-D, non-square, transposed);
 * a one-wave schedule for small depthwise problems; and two tensor-core
 * depthwise schedules (banded weight matrices) for NCHW and channels-last
 * 16-bit tensors.  GCONV_SCHED_AUTO lets the per-shape picker choose. */
typedef enum gconv_schedule {
    GCONV_SCHED_AUTO = -1,
    GCONV_SCHED_DW_FLAT = 0,     /* fallback: any layout, multiplier and group shape */
    GCONV_SCHED_DW_ROW8 = 1,     /* channels-last depthwise, square 3/5/7 kernel, stride 1
                                    or 2: input rows streamed through shared memory by TMA,
                                    register sliding window down the rows; also the
                                    stride-2 transposed form (a gather over the same ring) */
    GCONV_SCHED_DW_MULT = 2,     /* depthwise, multiplier <= 16: every output channel of an
                                    input channel from one input load */
    GCONV_SCHED_GRP_PLANE = 3,   /* grouped: a block per (image, group, tile), the group's
                                    weights shared in shared memory */
    GCONV_SCHED_GRP_REDUCE = 4,  /* grouped, few outputs: taps split across the lanes of a
                                    warp and reduced with shuffles */
    GCONV_SCHED_GRP_TC = 5,      /* grouped, 4 or 8 channels per group, channels-last bf16 /
                                    fp16: implicit GEMM on the tcgen05 tensor cores, fp32
                                    accumulation in tensor memory */
    GCONV_SCHED_DW_LINE = 6,     /* channels-last depthwise (multiplier 1), any kernel shape,
                                    stride and dilation, forward or transposed: a thread per
                                    16-byte channel vector and strip of output pixels */
    GCONV_SCHED_DW_SMALL = 7,    /* depthwise (any multiplier, layout, stride, dilation),
                                    forward: one pass, a thread per 4 outputs of a row, no
                                    shared memory; picked for NCHW problems of <= 2^20
                                    outputs */
    GCONV_SCHED_DW_TC = 8,       /* NCHW bf16 / fp16 depthwise (multiplier 1, 2, 4, 8 or 16)
                                    at stride 1: input rows times banded weight matrices on
                                    the tcgen05 tensor cores, fp32 accumulation in tensor
                                    memory */
    GCONV_SCHED_DW_TCL = 9,      /* channels-last bf16 / fp16 depthwise (multiplier 1) at
                                    stride 1, channels a multiple of 8: the input transposed
                                    to channel planes in shared memory, rows times banded
                                    weight matrices on the tcgen05 tensor cores; picked for
                                    2-D kernels outside dw_row8's with >= 12 taps */
    GCONV_SCHED_COUNT = 10
} gconv_schedule;

typedef enum gconv_layout {
    GCONV_LAYOUT_NCHW = 0,
    GCONV_LAYOUT_NHWC = 1        /* channels-last */
} gconv_layout;

/* A tensor's geometry: logical sizes and element strides.  x is [N, C, H, W]
 * (or [C, H, W] when unbatched), w is [C_out, C_in/groups, KH, KW], bias is
 * [C_out].  Strides are in elements, in the same logical order. */
typedef struct gconv_tensor {
    int32_t rank;
    int64_t sizes[4];
    int64_t strides[4];
} gconv_tensor;

/* The canonical, validated description of one convolution, filled by
 * conv_bind (or conv1d_bind, conv_transpose_bind, conv_transpose1d_bind).
 * Callers may change only `schedule` (GCONV_SCHED_AUTO or a gconv_schedule
 * value to force one schedule for calls with this desc).
 * A 1-D convolution is described as the 2-D one of height 1 (H = KH = OH =
 * 1, stride_h = dil_h = 1, no padding along h); for a transposed one, w is
 * [C_in, C_out/groups, KH, KW] and w_strides follow that order, H x W is
 * the input's size and OH x OW the output's, pad_before / pad_after are the
 * crops before and after, and output_padding extends the end. */
typedef struct gconv_desc {
    uint32_t magic;              /* set by conv_bind */
    int32_t dtype;               /* gconv_dtype */
    int32_t layout;              /* gconv_layout of x; y uses the same */
    int32_t has_bias;
    int32_t unbatched;           /* x was rank 3: y is rank 3 too */
    int32_t schedule;            /* GCONV_SCHED_AUTO unless forced by the caller */
    int64_t N, C_in, H, W;
    int64_t C_out, groups, Cin_g, Cout_g;
    int64_t KH, KW, OH, OW;
    int32_t stride[2];           /* (h, w) */
    int32_t pad_before[2];       /* (h, w) */
    int32_t pad_after[2];        /* (h, w) */
    int64_t x_strides[4];        /* elements, logical (N, C, H, W) order */
    int64_t w_strides[4];        /* elements, logical (C_out, Cin_g, KH, KW) order */
    int64_t b_stride;            /* elements; 0 when there is no bias */
    int64_t y_strides[4];        /* dense in `layout`, logical (N, C_out, OH, OW) order */
    int32_t x_dense;             /* x is dense (no gaps) in its layout */
    int32_t transposed;          /* 1: transposed convolution */
    int32_t spatial_dims;        /* 2, or 1 for conv1d_bind / conv_transpose1d_bind */
    int32_t reserved;
    int32_t dilation[2];         /* (h, w), >= 1 */
    int32_t output_padding[2];   /* (h, w), transposed only; 0 otherwise */
} gconv_desc;

/* Validate the arguments of one convolution and canonicalise them into *out
 * (the binding step of PR #25084, second paragraph: defaults filled, rank-3
 * input treated as one image -- torch/_inductor/kernel/conv.py, convolution,
 * adds the batch dim the same way -- and the group shape checked as
 * C_in == Cin_g * groups).
 *   x, w:        required geometries; bias: NULL for no bias.
 *   dtype:       gconv_dtype shared by x, w, bias and y.
 *   stride, padding_before, padding_after, dilation: (h, w) pairs; NULL
 *                stride/dilation mean 1, NULL paddings mean 0.  Dilation d
 *                spaces the taps d apart, so a window spans d*(K-1)+1 input
 *                positions and OH = floor((H + pb + pa - d*(KH-1) - 1) /
 *                stride_h) + 1.
 *   groups:      >= 1, divides C_in and C_out.
 * x must be NCHW-ordered (W stride 1, then H, then C, then N, no overlap) or
 * channels-last-ordered (C stride 1, then W, then H, then N); dims of size 1
 * are ignored, and when both orders fit NCHW is taken.  Pure host code: no
 * CUDA call.  Returns GCONV_OK or the first violated rule's status. */
gconv_status conv_bind(const gconv_tensor *x, const gconv_tensor *w,
                       const gconv_tensor *bias, int32_t dtype,
                       const int32_t stride[2], const int32_t padding_before[2],
                       const int32_t padding_after[2], const int32_t dilation[2],
                       int64_t groups, gconv_desc *out);

/* 1-D convolution (PR #25084, first paragraph, names 1-D convolutions among
 * the calls Inductor's templates cannot compile): x is [N, C_in, L] (or
 * [C_in, L], one sequence), w [C_out, Cin_g, K], bias [C_out]; stride,
 * padding and dilation are scalars along L.  x must be NCL-ordered (L
 * stride 1) or NLC-ordered (channels-last: C stride 1).  The desc is the
 * height-1 2-D convolution (spatial_dims = 1); out_shape_and_stride gives
 * [N, C_out, OL] (or [C_out, OL]), dense in x's order, and the forward entry
 * points run it as they run 2-D calls.  Same errors as conv_bind. */
gconv_status conv1d_bind(const gconv_tensor *x, const gconv_tensor *w,
                         const gconv_tensor *bias, int32_t dtype, int32_t stride,
                         int32_t padding_before, int32_t padding_after,
                         int32_t dilation, int64_t groups, gconv_desc *out);

/* Transposed 2-D convolution (executorch PR #25091, second paragraph): the
 * output pixel o reads, at tap k, the input (o + padding_before - k*d) /
 * stride whenever that is a whole number inside the input, with the weight
 * w [C_in, C_out/groups, KH, KW] (the forward weight's first two dims
 * swapped):
 *   y[n, co, oh, ow] = b[co] + sum_{ci, kh, kw} w[g*Cin_g + ci, co - g*Cout_g, kh, kw]
 *                               * x[n, g*Cin_g + ci, ih, iw],
 *   ih = (oh + pad_before_h - kh*dil_h) / stride_h (a whole number in [0, H)),
 *   iw likewise.
 * OH = (H - 1)*stride_h + dil_h*(KH - 1) + 1 + output_padding_h
 *      - padding_before_h - padding_after_h  (the uncropped output, extended
 * by output_padding at the end, cropped by the two paddings -- asymmetric
 * crops allowed); OH < 1 is GCONV_ERR_PADDING.  0 <= output_padding.
 * Envelope: KH, KW in [1, 9], Cin_g = C_in/groups <= 8 (the direct-stencil
 * bound, read on the transposed input side), any stride and dilation.
 * x layout, unbatched rank-3 input and the output layout follow conv_bind.
 * Run it with conv_transpose_forward. */
gconv_status conv_transpose_bind(const gconv_tensor *x, const gconv_tensor *w,
                                 const gconv_tensor *bias, int32_t dtype,
                                 const int32_t stride[2], const int32_t padding_before[2],
                                 const int32_t padding_after[2],
                                 const int32_t output_padding[2], const int32_t dilation[2],
                                 int64_t groups, gconv_desc *out);

/* Transposed 1-D convolution: x [N, C_in, L] (or [C_in, L]), w [C_in,
 * C_out/groups, K]; the height-1 case of conv_transpose_bind (PR #25091's
 * benchmark adds 1-D transposed upsampling, kernel 4 stride 2). */
gconv_status conv_transpose1d_bind(const gconv_tensor *x, const gconv_tensor *w,
                                   const gconv_tensor *bias, int32_t dtype,
                                   int32_t stride, int32_t padding_before,
                                   int32_t padding_after, int32_t output_padding,
                                   int32_t dilation, int64_t groups, gconv_desc *out);

/* The output's rank, sizes and element strides (PR #25084, second paragraph:
 * one function decides the output layout and both the op and its shape-only
 * variant use it).  Forward: OH = floor((H + pad_before_h + pad_after_h -
 * dilation_h * (KH - 1) - 1) / stride_h) + 1 and likewise OW (with
 * dilation 1: floor((H + pad_before_h + pad_after_h - KH) / stride_h) + 1);
 * transposed: the size conv_transpose_bind states.  y is dense in the layout of x
 * (NCHW in -> NCHW out, channels-last in -> channels-last out) and rank 3
 * when x was rank 3.  Pure host code. */
gconv_status out_shape_and_stride(const gconv_desc *d, int32_t *rank,
                                  int64_t sizes[4], int64_t strides[4]);

/* Depthwise forward (Cin_g == 1, any multiplier C_out / C_in).  Takes a
 * forward desc (conv_bind or conv1d_bind); a transposed one is
 * GCONV_ERR_KIND.  x, w, bias
 * and y are device pointers laid out as the geometries given to conv_bind
 * and as out_shape_and_stride says for y; bias must be NULL exactly when the
 * desc has none.  Launches on `stream` and returns without waiting.  Empty
 * problems (N, C_out, OH or OW zero) return GCONV_OK without a launch.
 * Returns GCONV_ERR_UNSUPPORTED when Cin_g != 1. */
gconv_status conv_dw_forward(const gconv_desc *d, const void *x, const void *w,
                             const void *bias, void *y, gconv_stream stream);

/* Grouped forward (1 <= Cin_g <= 8, any Cout_g); accepts depthwise descs
 * too.  Same pointer, stream and error contract as conv_dw_forward. */
gconv_status conv_grouped_forward(const gconv_desc *d, const void *x,
                                  const void *w, const void *bias, void *y,
                                  gconv_stream stream);

/* Transposed forward: runs a desc from conv_transpose_bind or
 * conv_transpose1d_bind (a forward desc is GCONV_ERR_KIND).  Pointers,
 * stream and errors as conv_dw_forward; w is [C_in, C_out/groups, KH, KW]
 * by the strides given to the bind.  A stride-1 transposed convolution
 * with one input or one output channel per group is the forward convolution
 * with the kernel flipped and padding d*(K-1) - crop, and runs on the
 * forward schedules; the others run on dw_line (channels-last depthwise),
 * or grp_reduce / dw_flat. */
gconv_status conv_transpose_forward(const gconv_desc *d, const void *x, const void *w,
                                    const void *bias, void *y, gconv_stream stream);

/* Timed schedule choice (PR #25085, second paragraph: the template's
 * schedules are timed at compile time and the fastest is used).  Runs every
 * schedule that takes this call (forward or transposed desc) once to warm
 * up and then `reps` times on `stream`, times each with CUDA events, and
 * records the fastest for the call's shape: later calls whose desc has
 * GCONV_SCHED_AUTO (and no process-wide override) with the same shape,
 * dtype, layout, strides and pointer alignment run it.  Unlike the other
 * entry points it waits for the stream (to read the events) and creates
 * and destroys two CUDA events; it writes y (the chosen schedule runs
 * last, so y holds its result).  *schedule gets the choice and *us its
 * time per launch in microseconds (either may be NULL).  reps < 1 is
 * GCONV_ERR_SHAPE; the record is process-wide and guarded by a mutex. */
gconv_status conv_autotune(const gconv_desc *d, const void *x, const void *w, const void *bias,
                           void *y, gconv_stream stream, int32_t reps, int32_t *schedule,
                           float *us);

/* Forget every schedule conv_autotune recorded. */
void conv_autotune_clear(void);

/* Which schedule a forward call with this desc and these pointers would run
 * (the picker, or the forced schedule), without launching anything.  Pointer
 * values are only inspected for alignment.  Returns GCONV_ERR_SCHEDULE /
 * GCONV_ERR_ALIGN when a forced schedule cannot run the call. */
gconv_status conv_select_schedule(const gconv_desc *d, const void *x,
                                  const void *w, const void *bias,
                                  const void *y, int32_t *schedule);

/* ---------------------------------------------------------------- backward
 * The gradients of the forward convolution described by a forward desc d
 * (torch/_inductor/kernel/conv.py, convolution_backward_lowering: grad
 * input, grad weight, and grad bias = the sum of grad_output over batch and
 * space).  gy, the output gradient, has the sizes and strides that
 * out_shape_and_stride gives for y. */

/* Sizes and strides of dx: x's sizes, dense in x's layout (NCHW or
 * channels-last; rank 3 / 2 for unbatched or 1-D descs, as x was). */
gconv_status grad_input_shape_and_stride(const gconv_desc *d, int32_t *rank,
                                         int64_t sizes[4], int64_t strides[4]);

/* dx = the gradient of sum(y * gy) with respect to x: every forward product
 * w * x sends gy * w to dx at x's index.  It is the transposed convolution
 * of gy with the forward weight (same stride, dilation and groups, crop
 * pad_before, sized back to H x W), and runs on the transposed schedules.
 * gy, w, dx are device pointers (dx laid out as grad_input_shape_and_stride
 * says); fp32 accumulation, one rounding to the dtype.  Same stream and error
 * contract as the forward. */
gconv_status conv_backward_input(const gconv_desc *d, const void *gy, const void *w,
                                 void *dx, gconv_stream stream);

/* Bytes of device workspace conv_backward_weight needs for this desc (the
 * fp32 partial sums of its first pass).  Pure host code. */
gconv_status conv_backward_weight_workspace_size(const gconv_desc *d, uint64_t *bytes);

/* dw[co, ci, kh, kw] = sum over n, oh, ow of gy[n, co, oh, ow] * x[n, g*Cin_g + ci, ih, iw]
 * (the taps of the forward), written dense [C_out, Cin_g, KH, KW] in the
 * dtype; db[co] = sum over n, oh, ow of gy[n, co, oh, ow], dense [C_out]
 * (db may be NULL to skip it).  Two launches: partial sums over slices of
 * the output pixels in fp32 into `workspace` (at least the bytes
 * conv_backward_weight_workspace_size gives, 16-byte aligned, owned by the
 * caller and not read before it is written), then a pass that adds the
 * slices in a fixed order (compensated fp32 sums, as accurate as twice the
 * precision) and rounds once.  The result is deterministic.  x and gy as
 * for the forward and conv_backward_input. */
gconv_status conv_backward_weight(const gconv_desc *d, const void *x, const void *gy,
                                  void *dw, void *db, void *workspace,
                                  uint64_t workspace_bytes, gconv_stream stream);

/* conv_backward_weight without a caller workspace, for callers that cannot
 * allocate device memory: code inside a host framework that owns every
 * device allocation (only its pool may be used, and this library has no
 * handle to it), or code on a fixed memory budget that allows no allocation
 * after start-up.  The pages have no counterpart; the computation and the
 * result are those of conv_backward_weight (same kernels, bit for bit).
 * Its scratch is a fixed buffer of conv_backward_weight_noalloc_limit()
 * bytes (8 MiB) in device memory, which every GPU that loads the library
 * holds until the process exits; a problem whose
 * conv_backward_weight_workspace_size exceeds it gets
 * GCONV_ERR_SCRATCH_LIMIT.  The first call with a device current looks the
 * buffer's address up on that device (make it before any stream capture
 * begins) and keeps it for the life of the process, so the device must not
 * be reset (cudaDeviceReset) while the library is in use.  The call itself
 * allocates nothing.  All calls share the buffer:
 * each writes every scratch entry before reading it, so no clearing is
 * needed, but calls whose kernels overlap on the GPU race on it -- keep
 * them ordered on one stream. */
gconv_status conv_backward_weight_noalloc(const gconv_desc *d, const void *x, const void *gy,
                                          void *dw, void *db, gconv_stream stream);

/* Size in bytes of conv_backward_weight_noalloc's fixed device buffer. */
uint64_t conv_backward_weight_noalloc_limit(void);

/* Process-wide override for tests (the force_conv_candidate hook of PR
 * #25084): every later call whose desc has schedule == GCONV_SCHED_AUTO runs
 * `schedule`, or the picker again when GCONV_SCHED_AUTO.  The environment
 * variable GCONV_FORCE_SCHEDULE (a schedule name or number) sets the initial
 * value.  Returns GCONV_ERR_SCHEDULE for an unknown value. */
gconv_status conv_force_schedule(int32_t schedule);

/* Name of a schedule ("dw_flat", ...), or "auto" / "unknown". */
const char *conv_schedule_name(int32_t schedule);

/* Human-readable text for a status. */
const char *conv_strerror(gconv_status status);

/* Test hook for the failure path: when `cuda_error` is non-zero, the next
 * forward call that would launch returns GCONV_ERR_CUDA without launching,
 * exactly as if the launch had failed with that error; 0 clears it.  Lets the
 * error path be tested without making a GPU fail. */
void conv_test_inject_launch_error(int32_t cuda_error);

/* The CUDA error code behind the last GCONV_ERR_CUDA returned on this host
 * thread (0 if none). */
int32_t conv_last_cuda_error(void);

/* Number of kernels this library has launched in this process (all
 * threads).  Lets callers count launches inside a timed region. */
uint64_t conv_launch_count(void);

/* Measurement aid, not part of the convolution: launches one kernel of
 * independent fp32 FMA chains sized to fill every SM (`trips` loop trips of
 * 128 FMAs per thread) on `stream` and returns in *fmas the number of FMAs
 * it performs, so the caller can time it with events and state the chip's
 * FP32 FMA rate, the roofline of the FMA-bound stencils.  `sink` is a
 * device buffer of at least (SMs x resident blocks) floats that the kernel
 * may write (it never does for finite inputs).  Errors: GCONV_ERR_NULL,
 * GCONV_ERR_SHAPE (trips < 1), GCONV_ERR_CUDA. */
gconv_status conv_probe_fma_rate(int32_t trips, float *sink, gconv_stream stream,
                                 uint64_t *fmas);

/* Library version as major*10000 + minor*100 + patch. */
int32_t conv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GCONV_H */
