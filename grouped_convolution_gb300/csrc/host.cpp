// host.cpp -- the host half of the C ABI: argument binding and validation,
// the output layout, the per-shape schedule picker and the forward entry
// points.  Nothing here allocates device memory or synchronises.
//
// Binding follows the canonical convolution op of executorch PR #25084 "Add
// triton::convolution and the conv routing framework" (description, second
// paragraph): every call is mapped to one canonical form with explicit
// padding before and after, defaults filled and arguments validated; one
// function computes the output layout; the output is allocated once by the
// caller and the kernels only write into it.  The accepted envelope is the
// direct-stencil template's, executorch PR #25085 (description, second
// paragraph).

#include <atomic>
#include <climits>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <vector>

#include "gconv_internal.h"

using namespace gconv;

namespace {

std::atomic<int32_t> g_forced{INT32_MIN};   // INT32_MIN: not yet read from env
std::atomic<int32_t> g_inject{0};
std::atomic<uint64_t> g_launches{0};
thread_local int32_t t_last_cuda_error = 0;

const Schedule *const kSchedules[GCONV_SCHED_COUNT] = {
    &kDwFlat, &kDwRow8, &kDwMult, &kGrpPlane, &kGrpReduce, &kGrpTc, &kDwLine, &kDwSmall, &kDwTc, &kDwTcl};

}  // namespace

namespace gconv {
bool pdl_enabled() {
    static const bool on = [] {
        const char *e = std::getenv("GCONV_PDL");
        return e && e[0] == '1' && e[1] == 0;
    }();
    return on;
}
}  // namespace gconv

namespace {

int32_t schedule_from_string(const char *s) {
    if (!s || !*s) return GCONV_SCHED_AUTO;
    if (!strcmp(s, "auto")) return GCONV_SCHED_AUTO;
    for (int i = 0; i < GCONV_SCHED_COUNT; ++i)
        if (!strcmp(s, kSchedules[i]->name)) return i;
    char *end = nullptr;
    long v = strtol(s, &end, 10);
    if (end && *end == '\0' && v >= -1 && v < GCONV_SCHED_COUNT) return (int32_t)v;
    return GCONV_SCHED_AUTO;
}

int32_t forced_schedule() {
    int32_t f = g_forced.load(std::memory_order_relaxed);
    if (f == INT32_MIN) {
        int32_t env = schedule_from_string(getenv("GCONV_FORCE_SCHEDULE"));
        int32_t expect = INT32_MIN;
        g_forced.compare_exchange_strong(expect, env);
        f = g_forced.load(std::memory_order_relaxed);
    }
    return f;
}

bool fits_i32(int64_t v) { return v >= 0 && v <= INT32_MAX; }

// Dense element strides of an [N, C, H, W] tensor in a layout.
void dense_strides(int32_t layout, int64_t N, int64_t C, int64_t H, int64_t W,
                   int64_t st[4]) {
    (void)N;
    if (layout == GCONV_LAYOUT_NCHW) {
        st[3] = 1; st[2] = W; st[1] = H * W; st[0] = C * H * W;
    } else {
        st[1] = 1; st[3] = C; st[2] = W * C; st[0] = H * W * C;
    }
}

// Rank, sizes and strides of an [N, C, H, W] tensor as the caller sees it:
// rank 4 (2-D), 3 (1-D: [N, C, L]), one less when unbatched.
void user_geometry(const gconv_desc &d, const int64_t s4[4], const int64_t t4[4],
                   int32_t *rank, int64_t sizes[4], int64_t strides[4]) {
    int64_t s[4], t[4];
    int r = 0;
    for (int i = 0; i < 4; ++i) {
        if (i == 0 && d.unbatched) continue;
        if (i == 2 && d.spatial_dims == 1) continue;
        s[r] = s4[i]; t[r] = t4[i]; ++r;
    }
    *rank = r;
    for (int i = 0; i < 4; ++i) {
        sizes[i] = i < r ? s[i] : 0;
        strides[i] = i < r ? t[i] : 0;
    }
}

// Dims with size 1 are ignored; remaining dims must appear with strictly
// nesting strides in `order` (outermost first) and the innermost has
// stride 1.  Sets *dense when the strides are exactly the dense ones.
bool ordered(const int64_t sizes[4], const int64_t strides[4], const int order[4],
             bool *dense) {
    int64_t inner_extent = 1;   // elements spanned by the dims inside the current one
    bool first = true;
    *dense = true;
    for (int k = 3; k >= 0; --k) {
        int d = order[k];
        if (sizes[d] == 1) continue;
        if (sizes[d] == 0) continue;
        if (first) {
            if (strides[d] != 1) return false;
            first = false;
        } else {
            if (strides[d] < inner_extent) return false;
            if (strides[d] != inner_extent) *dense = false;
        }
        inner_extent = strides[d] * sizes[d];
    }
    return true;
}

}  // namespace

namespace gconv {

void note_launches(int launches) {
    g_launches.fetch_add((uint64_t)launches, std::memory_order_relaxed);
}

void note_cuda_error(int32_t e) { t_last_cuda_error = e; }

// The injected-error hook of conv_test_inject_launch_error: a pending value
// makes this call fail as a launch error would, without launching.
gconv_status take_injected() {
    int32_t inj = g_inject.exchange(0);
    if (inj != 0) {
        t_last_cuda_error = inj;
        return GCONV_ERR_CUDA;
    }
    return GCONV_OK;
}

Params make_params(const gconv_desc &d) {
    Params p{};
    p.N = (int)d.N; p.C_in = (int)d.C_in; p.H = (int)d.H; p.W = (int)d.W;
    p.C_out = (int)d.C_out; p.G = (int)d.groups; p.Cin_g = (int)d.Cin_g;
    p.Cout_g = (int)d.Cout_g; p.KH = (int)d.KH; p.KW = (int)d.KW;
    p.OH = (int)d.OH; p.OW = (int)d.OW;
    p.sh = d.stride[0]; p.sw = d.stride[1];
    p.pbh = d.pad_before[0]; p.pbw = d.pad_before[1];
    p.dh = d.dilation[0]; p.dw = d.dilation[1];
    p.transposed = d.transposed;
    p.has_bias = d.has_bias; p.layout = d.layout; p.dtype = d.dtype;
    for (int i = 0; i < 4; ++i) {
        p.xs[i] = d.x_strides[i]; p.ws[i] = d.w_strides[i]; p.ys[i] = d.y_strides[i];
    }
    p.bs = d.b_stride;
    return p;
}

}  // namespace gconv

namespace {

// A call of any binding entry point, in canonical rank-4 form: x [N, C, H,
// W], w [C_out, Cin_g, KH, KW] (forward) or [C_in, Cout_g, KH, KW]
// (transposed); 1-D calls have H = KH = 1.
struct BindArgs {
    int64_t xs[4], xst[4], ws[4], wst[4];
    int unbatched, spatial_dims, transposed;
    const gconv_tensor *bias;
    int32_t dtype;
    int32_t st[2], pb[2], pa[2], dil[2], op[2];
    int64_t groups;
};

gconv_status bind_common(const BindArgs &a, gconv_desc *out) {
    gconv_desc d;
    memset(&d, 0, sizeof(d));
    for (int i = 0; i < 4; ++i) {
        if (a.xs[i] < 0 || a.ws[i] < 0) return GCONV_ERR_SHAPE;
        if (!fits_i32(a.xs[i]) || !fits_i32(a.ws[i])) return GCONV_ERR_UNSUPPORTED;
        if (a.xst[i] < 0 || a.wst[i] < 0) return GCONV_ERR_LAYOUT;
    }
    const int64_t N = a.xs[0], C_in = a.xs[1], H = a.xs[2], W = a.xs[3];
    const int64_t KH = a.ws[2], KW = a.ws[3];
    const int64_t groups = a.groups;
    if (groups < 1) return GCONV_ERR_SHAPE;
    int64_t C_out, Cin_g;
    if (!a.transposed) {
        // Group shape: C_in == Cin_g * groups (torch/_inductor/kernel/conv.py,
        // convolution: in_chan * groups == C_in), groups divides C_out.
        C_out = a.ws[0];
        Cin_g = a.ws[1];
        if (Cin_g < 1 || Cin_g * groups != C_in) return GCONV_ERR_SHAPE;
        if (C_out % groups != 0) return GCONV_ERR_SHAPE;
    } else {
        // The transposed weight is [C_in, C_out / groups, KH, KW].
        if (a.ws[0] != C_in || C_in % groups != 0) return GCONV_ERR_SHAPE;
        Cin_g = C_in / groups;
        C_out = a.ws[1] * groups;
        if (Cin_g < 1 && C_in > 0) return GCONV_ERR_SHAPE;
        if (!fits_i32(C_out)) return GCONV_ERR_UNSUPPORTED;
    }
    if (a.bias) {
        if (a.bias->sizes[0] != C_out) return GCONV_ERR_SHAPE;
        if (a.bias->strides[0] < 0) return GCONV_ERR_LAYOUT;
    }
    if (a.st[0] < 1 || a.st[1] < 1) return GCONV_ERR_SHAPE;

    // The envelope: kernels up to 9x9, at most 8 input channels per group
    // (PR #25085); any dilation >= 1.
    if (a.dil[0] < 1 || a.dil[1] < 1) return GCONV_ERR_UNSUPPORTED;
    if (KH < 1 || KH > 9 || KW < 1 || KW > 9) return GCONV_ERR_UNSUPPORTED;
    if (Cin_g > 8) return GCONV_ERR_UNSUPPORTED;

    if (a.pb[0] < 0 || a.pb[1] < 0 || a.pa[0] < 0 || a.pa[1] < 0) return GCONV_ERR_PADDING;
    if (a.op[0] < 0 || a.op[1] < 0) return GCONV_ERR_PADDING;
    const int64_t span_h = (int64_t)a.dil[0] * (KH - 1) + 1;
    const int64_t span_w = (int64_t)a.dil[1] * (KW - 1) + 1;
    int64_t OH, OW;
    if (!a.transposed) {
        const int64_t Hp = H + a.pb[0] + a.pa[0], Wp = W + a.pb[1] + a.pa[1];
        if (Hp < span_h || Wp < span_w) return GCONV_ERR_PADDING;
        OH = (Hp - span_h) / a.st[0] + 1;
        OW = (Wp - span_w) / a.st[1] + 1;
    } else {
        // Uncropped output (H - 1) * s + span, extended by output_padding,
        // cropped by the paddings.  An empty input has no output extent.
        if (H < 1 || W < 1) return GCONV_ERR_SHAPE;
        OH = (H - 1) * a.st[0] + span_h + a.op[0] - a.pb[0] - a.pa[0];
        OW = (W - 1) * a.st[1] + span_w + a.op[1] - a.pb[1] - a.pa[1];
        if (OH < 1 || OW < 1) return GCONV_ERR_PADDING;
    }
    if (!fits_i32(OH) || !fits_i32(OW)) return GCONV_ERR_UNSUPPORTED;

    // Layout of x: NCHW-ordered or channels-last-ordered; NCHW on a tie.
    static const int kNCHW[4] = {0, 1, 2, 3}, kNHWC[4] = {0, 2, 3, 1};
    bool dense_nchw = false, dense_nhwc = false;
    if (ordered(a.xs, a.xst, kNCHW, &dense_nchw)) {
        d.layout = GCONV_LAYOUT_NCHW;
        d.x_dense = dense_nchw;
    } else if (ordered(a.xs, a.xst, kNHWC, &dense_nhwc)) {
        d.layout = GCONV_LAYOUT_NHWC;
        d.x_dense = dense_nhwc;
    } else {
        return GCONV_ERR_LAYOUT;
    }

    // Size products must stay far from int64 overflow.
    const double big = 4.0e18;
    if ((double)N * C_out * OH * OW > big || (double)N * C_in * H * W > big)
        return GCONV_ERR_UNSUPPORTED;

    d.dtype = a.dtype;
    d.has_bias = a.bias != nullptr;
    d.unbatched = a.unbatched;
    d.transposed = a.transposed;
    d.spatial_dims = a.spatial_dims;
    d.schedule = GCONV_SCHED_AUTO;
    d.N = N; d.C_in = C_in; d.H = H; d.W = W;
    d.C_out = C_out; d.groups = groups; d.Cin_g = Cin_g; d.Cout_g = C_out / groups;
    d.KH = KH; d.KW = KW; d.OH = OH; d.OW = OW;
    for (int i = 0; i < 2; ++i) {
        d.stride[i] = a.st[i];
        d.pad_before[i] = a.pb[i];
        d.pad_after[i] = a.pa[i];
        d.dilation[i] = a.dil[i];
        d.output_padding[i] = a.transposed ? a.op[i] : 0;
    }
    for (int i = 0; i < 4; ++i) { d.x_strides[i] = a.xst[i]; d.w_strides[i] = a.wst[i]; }
    d.b_stride = a.bias ? a.bias->strides[0] : 0;
    dense_strides(d.layout, N, C_out, OH, OW, d.y_strides);
    d.magic = kDescMagic;
    *out = d;
    return GCONV_OK;
}

// Rank-4 x geometry from a rank-3/4 tensor (2-D calls) or rank-2/3 (1-D).
gconv_status canon_x(const gconv_tensor *x, int spatial_dims, BindArgs &a) {
    const int r = x->rank;
    if (spatial_dims == 2) {
        if (r != 3 && r != 4) return GCONV_ERR_RANK;
        const int off = 4 - r;
        a.xs[0] = 1; a.xst[0] = 0;
        for (int i = 0; i < r; ++i) { a.xs[i + off] = x->sizes[i]; a.xst[i + off] = x->strides[i]; }
        a.unbatched = r == 3;
    } else {
        if (r != 2 && r != 3) return GCONV_ERR_RANK;
        const int off = 3 - r;
        int64_t s3[3] = {1, 0, 0}, t3[3] = {0, 0, 0};
        for (int i = 0; i < r; ++i) { s3[i + off] = x->sizes[i]; t3[i + off] = x->strides[i]; }
        a.xs[0] = s3[0]; a.xst[0] = t3[0];
        a.xs[1] = s3[1]; a.xst[1] = t3[1];
        a.xs[2] = 1;     a.xst[2] = t3[2] * (s3[2] > 0 ? s3[2] : 1);  // height 1: stride unused
        a.xs[3] = s3[2]; a.xst[3] = t3[2];
        a.unbatched = r == 2;
    }
    return GCONV_OK;
}

gconv_status canon_w(const gconv_tensor *w, int spatial_dims, BindArgs &a) {
    if (spatial_dims == 2) {
        if (w->rank != 4) return GCONV_ERR_RANK;
        for (int i = 0; i < 4; ++i) { a.ws[i] = w->sizes[i]; a.wst[i] = w->strides[i]; }
    } else {
        if (w->rank != 3) return GCONV_ERR_RANK;
        a.ws[0] = w->sizes[0]; a.wst[0] = w->strides[0];
        a.ws[1] = w->sizes[1]; a.wst[1] = w->strides[1];
        a.ws[2] = 1;           a.wst[2] = w->strides[2] * (w->sizes[2] > 0 ? w->sizes[2] : 1);
        a.ws[3] = w->sizes[2]; a.wst[3] = w->strides[2];
    }
    return GCONV_OK;
}

gconv_status bind_entry(const gconv_tensor *x, const gconv_tensor *w, const gconv_tensor *bias,
                        int32_t dtype, int spatial_dims, int transposed, const int32_t st[2],
                        const int32_t pb[2], const int32_t pa[2], const int32_t dil[2],
                        const int32_t op[2], int64_t groups, gconv_desc *out) {
    if (!x || !w || !out) return GCONV_ERR_NULL;
    if (dtype != GCONV_F32 && dtype != GCONV_F16 && dtype != GCONV_BF16) return GCONV_ERR_DTYPE;
    if (bias && bias->rank != 1) return GCONV_ERR_RANK;
    BindArgs a;
    memset(&a, 0, sizeof(a));
    gconv_status e = canon_x(x, spatial_dims, a);
    if (e != GCONV_OK) return e;
    e = canon_w(w, spatial_dims, a);
    if (e != GCONV_OK) return e;
    a.spatial_dims = spatial_dims;
    a.transposed = transposed;
    a.bias = bias;
    a.dtype = dtype;
    a.groups = groups;
    for (int i = 0; i < 2; ++i) {
        a.st[i] = st[i]; a.pb[i] = pb[i]; a.pa[i] = pa[i]; a.dil[i] = dil[i]; a.op[i] = op[i];
    }
    return bind_common(a, out);
}

}  // namespace

extern "C" {

gconv_status conv_bind(const gconv_tensor *x, const gconv_tensor *w,
                       const gconv_tensor *bias, int32_t dtype,
                       const int32_t stride[2], const int32_t padding_before[2],
                       const int32_t padding_after[2], const int32_t dilation[2],
                       int64_t groups, gconv_desc *out) {
    // NULL pointers take the canonical defaults.
    int32_t st[2] = {1, 1}, pb[2] = {0, 0}, pa[2] = {0, 0}, dil[2] = {1, 1}, op[2] = {0, 0};
    if (stride) { st[0] = stride[0]; st[1] = stride[1]; }
    if (padding_before) { pb[0] = padding_before[0]; pb[1] = padding_before[1]; }
    if (padding_after) { pa[0] = padding_after[0]; pa[1] = padding_after[1]; }
    if (dilation) { dil[0] = dilation[0]; dil[1] = dilation[1]; }
    return bind_entry(x, w, bias, dtype, 2, 0, st, pb, pa, dil, op, groups, out);
}

gconv_status conv1d_bind(const gconv_tensor *x, const gconv_tensor *w,
                         const gconv_tensor *bias, int32_t dtype, int32_t stride,
                         int32_t padding_before, int32_t padding_after,
                         int32_t dilation, int64_t groups, gconv_desc *out) {
    const int32_t st[2] = {1, stride}, pb[2] = {0, padding_before}, pa[2] = {0, padding_after},
                  dil[2] = {1, dilation}, op[2] = {0, 0};
    return bind_entry(x, w, bias, dtype, 1, 0, st, pb, pa, dil, op, groups, out);
}

gconv_status conv_transpose_bind(const gconv_tensor *x, const gconv_tensor *w,
                                 const gconv_tensor *bias, int32_t dtype,
                                 const int32_t stride[2], const int32_t padding_before[2],
                                 const int32_t padding_after[2],
                                 const int32_t output_padding[2], const int32_t dilation[2],
                                 int64_t groups, gconv_desc *out) {
    int32_t st[2] = {1, 1}, pb[2] = {0, 0}, pa[2] = {0, 0}, dil[2] = {1, 1}, op[2] = {0, 0};
    if (stride) { st[0] = stride[0]; st[1] = stride[1]; }
    if (padding_before) { pb[0] = padding_before[0]; pb[1] = padding_before[1]; }
    if (padding_after) { pa[0] = padding_after[0]; pa[1] = padding_after[1]; }
    if (output_padding) { op[0] = output_padding[0]; op[1] = output_padding[1]; }
    if (dilation) { dil[0] = dilation[0]; dil[1] = dilation[1]; }
    return bind_entry(x, w, bias, dtype, 2, 1, st, pb, pa, dil, op, groups, out);
}

gconv_status conv_transpose1d_bind(const gconv_tensor *x, const gconv_tensor *w,
                                   const gconv_tensor *bias, int32_t dtype,
                                   int32_t stride, int32_t padding_before,
                                   int32_t padding_after, int32_t output_padding,
                                   int32_t dilation, int64_t groups, gconv_desc *out) {
    const int32_t st[2] = {1, stride}, pb[2] = {0, padding_before}, pa[2] = {0, padding_after},
                  dil[2] = {1, dilation}, op[2] = {0, output_padding};
    return bind_entry(x, w, bias, dtype, 1, 1, st, pb, pa, dil, op, groups, out);
}

gconv_status out_shape_and_stride(const gconv_desc *d, int32_t *rank,
                                  int64_t sizes[4], int64_t strides[4]) {
    if (!d || !rank || !sizes || !strides) return GCONV_ERR_NULL;
    if (d->magic != kDescMagic) return GCONV_ERR_INTERNAL;
    const int64_t s4[4] = {d->N, d->C_out, d->OH, d->OW};
    user_geometry(*d, s4, d->y_strides, rank, sizes, strides);
    return GCONV_OK;
}

gconv_status grad_input_shape_and_stride(const gconv_desc *d, int32_t *rank,
                                         int64_t sizes[4], int64_t strides[4]) {
    if (!d || !rank || !sizes || !strides) return GCONV_ERR_NULL;
    if (d->magic != kDescMagic) return GCONV_ERR_INTERNAL;
    if (d->transposed) return GCONV_ERR_KIND;
    const int64_t s4[4] = {d->N, d->C_in, d->H, d->W};
    int64_t t4[4];
    dense_strides(d->layout, d->N, d->C_in, d->H, d->W, t4);
    user_geometry(*d, s4, t4, rank, sizes, strides);
    return GCONV_OK;
}

// The per-shape picker.  Specialised schedules win where they apply; the
// fallback schedule dw_flat takes everything else.  Small NCHW depthwise
// problems run on dw_small; larger NCHW 16-bit depthwise ones at stride 1 on
// the tensor cores (dw_tc).  Grouped calls the
// tensor cores can take (4 or 8 channels per group, channels-last 16-bit)
// run there.  Channels-last 16-bit 2-D depthwise calls at stride 1 whose
// kernels dw_row8 does not take run on the tensor cores (dw_tcl) when the
// kernel has at least 12 taps.  Other channels-last depthwise calls outside
// dw_row8's reach (1-D, small non-square kernels, fp32, dilation other than
// 2 on a stride-1 3x3, transposed calls other than stride 2) run on
// dw_line.  Other
// calls with too few outputs to give every thread of the GPU its own (fewer
// than 152 SMs x 512) and a long tap loop split the taps across lanes.
static int32_t pick(const gconv_desc &d, const Ptrs &p) {
    const bool dw = d.Cin_g == 1;
    // Depthwise NCHW problems of at most 2^20 outputs: one wave of threads
    // without a staging ring (its fill and drain cost more than the work).
    if (dw && d.layout == GCONV_LAYOUT_NCHW &&
        (double)d.N * d.C_out * d.OH * d.OW <= (double)(1 << 20) && kDwSmall.supports(d, p))
        return GCONV_SCHED_DW_SMALL;
    if (dw && d.Cout_g == 1 && kDwRow8.supports(d, p)) return GCONV_SCHED_DW_ROW8;
    // Channels-last 16-bit 2-D depthwise layers outside dw_row8's kernels
    // (even, 9x9 and non-square) at stride 1, with at least 12 taps: the
    // banded product on the tensor cores.  Measured on N 32, C 96, 56 x 56
    // bf16: 9x9 35 us against dw_line's 157, 8x8 34 / 130, 3x5 25 / 55,
    // 5x3 24 / 28, 4x4 25 / 26; but 2x2 23 / 15 and 1x1 23 / 11 (dw_tcl's
    // copies set a floor the small kernels' arithmetic never reaches).  1-D
    // layers stay on dw_line: their single rows leave most of a 128-row tile
    // empty.
    if (dw && d.Cout_g == 1 && d.spatial_dims == 2 && d.KH * d.KW >= 12 &&
        kDwTcl.supports(d, p))
        return GCONV_SCHED_DW_TCL;
    if (dw && kDwTc.supports(d, p)) return GCONV_SCHED_DW_TC;
    if (dw && kDwMult.supports(d, p)) return GCONV_SCHED_DW_MULT;
    if (!dw && kGrpTc.supports(d, p)) return GCONV_SCHED_GRP_TC;
    if (kDwLine.supports(d, p)) return GCONV_SCHED_DW_LINE;
    const double outputs = (double)d.N * d.C_out * d.OH * d.OW;
    const int64_t taps = d.Cin_g * d.KH * d.KW;
    if (outputs < 152.0 * 512 && taps >= 32) return GCONV_SCHED_GRP_REDUCE;
    if (kGrpPlane.supports(d, p)) return GCONV_SCHED_GRP_PLANE;
    return GCONV_SCHED_DW_FLAT;
}

// The schedule requested for a desc: its own, else the process-wide one.
static int32_t requested_schedule(const gconv_desc &d) {
    int32_t s = d.schedule;
    if (s == GCONV_SCHED_AUTO) s = forced_schedule();
    return s;
}

static gconv_status select_for(const gconv_desc &d, const Ptrs &p, int32_t s, int32_t *out) {
    if (s == GCONV_SCHED_AUTO) {
        *out = pick(d, p);
        return GCONV_OK;
    }
    if (s < 0 || s >= GCONV_SCHED_COUNT) return GCONV_ERR_SCHEDULE;
    if (!kSchedules[s]->supports(d, p)) {
        // Distinguish "this shape never runs here" from "these pointers are
        // not aligned enough": retry with ideally aligned pointers.
        Ptrs ideal{(const void *)(uintptr_t)4096, (const void *)(uintptr_t)4096,
                   p.b ? (const void *)(uintptr_t)4096 : nullptr, (void *)(uintptr_t)4096};
        return kSchedules[s]->supports(d, ideal) ? GCONV_ERR_ALIGN : GCONV_ERR_SCHEDULE;
    }
    *out = s;
    return GCONV_OK;
}

static bool empty_problem(const gconv_desc *d) {
    return d->N == 0 || d->C_out == 0 || d->OH == 0 || d->OW == 0;
}

static gconv_status check_call(const gconv_desc *d, const void *x, const void *w,
                               const void *bias, void *y) {
    if (!d) return GCONV_ERR_NULL;
    if (d->magic != kDescMagic) return GCONV_ERR_INTERNAL;
    // An empty problem touches no memory: its tensors may have NULL data.
    if (empty_problem(d)) return GCONV_OK;
    if (!x || !w || !y) return GCONV_ERR_NULL;
    if ((bias != nullptr) != (d->has_bias != 0)) return GCONV_ERR_NULL;
    return GCONV_OK;
}

// What one call runs: the desc the kernel sees (the caller's, or for a
// transposed call that is a flipped-kernel forward, that forward), its
// pointers and the schedule.
struct Plan {
    gconv_desc d;
    Ptrs p;
    int32_t schedule;
};

// A stride-1 transposed convolution is the forward convolution of the same
// input with the kernel flipped in both dims, padding d*(K-1) - crop before
// and d*(K-1) + output_padding - crop after (both must be >= 0):
//   y[o] = sum_k w[k] x[o + crop - k*d] = sum_k' w[K-1-k'] x[o - pad + k'*d].
// Output channel co = g*Cout_g + j reads weight w[g*Cin_g + ci, j]; that is a
// stride over (co, ci) when each group has one output channel (co stride
// Cin_g * ws0, ci stride ws0) or one input channel and nesting weight strides
// (co stride ws1).
static bool flipped_forward(const gconv_desc &t, const Ptrs &p, gconv_desc *f, Ptrs *q) {
    if (!t.transposed || t.stride[0] != 1 || t.stride[1] != 1) return false;
    int64_t co_stride, ci_stride;
    if (t.Cout_g == 1) {
        co_stride = t.Cin_g * t.w_strides[0];
        ci_stride = t.w_strides[0];
    } else if (t.Cin_g == 1 && t.w_strides[0] == t.Cout_g * t.w_strides[1]) {
        co_stride = t.w_strides[1];
        ci_stride = t.w_strides[0];   // one input channel: unused
    } else {
        return false;
    }
    const int64_t ext_h = (int64_t)t.dilation[0] * (t.KH - 1);
    const int64_t ext_w = (int64_t)t.dilation[1] * (t.KW - 1);
    const int64_t pbh = ext_h - t.pad_before[0], pbw = ext_w - t.pad_before[1];
    const int64_t pah = ext_h + t.output_padding[0] - t.pad_after[0];
    const int64_t paw = ext_w + t.output_padding[1] - t.pad_after[1];
    if (pbh < 0 || pbw < 0 || pah < 0 || paw < 0) return false;
    *f = t;
    f->transposed = 0;
    f->output_padding[0] = f->output_padding[1] = 0;
    f->pad_before[0] = (int32_t)pbh; f->pad_before[1] = (int32_t)pbw;
    f->pad_after[0] = (int32_t)pah; f->pad_after[1] = (int32_t)paw;
    f->w_strides[0] = co_stride;
    f->w_strides[1] = ci_stride;
    f->w_strides[2] = -t.w_strides[2];
    f->w_strides[3] = -t.w_strides[3];
    *q = p;
    q->w = static_cast<const char *>(p.w) +
           ((t.KH - 1) * t.w_strides[2] + (t.KW - 1) * t.w_strides[3]) * dtype_size(t.dtype);
    return true;
}

// Schedules chosen by conv_autotune, per call shape: every desc field that
// shapes the launch, and the pointers' alignment (which decides what the
// vectorised schedules take).
static std::mutex g_tuned_mutex;
static std::map<std::vector<int64_t>, int32_t> g_tuned;

static std::vector<int64_t> tune_key(const gconv_desc &d, const Ptrs &p) {
    std::vector<int64_t> k = {d.dtype, d.layout, d.transposed, d.spatial_dims, d.has_bias,
                              d.unbatched, d.N, d.C_in, d.H, d.W, d.C_out, d.groups, d.KH, d.KW,
                              d.stride[0], d.stride[1], d.pad_before[0], d.pad_before[1],
                              d.pad_after[0], d.pad_after[1], d.dilation[0], d.dilation[1],
                              d.output_padding[0], d.output_padding[1], d.b_stride};
    for (int i = 0; i < 4; ++i) {
        k.push_back(d.x_strides[i]);
        k.push_back(d.w_strides[i]);
        k.push_back(d.y_strides[i]);
    }
    const void *ptrs[4] = {p.x, p.w, p.b, p.y};
    for (const void *q : ptrs) k.push_back((int64_t)(reinterpret_cast<uintptr_t>(q) & 127));
    return k;
}

static int32_t tuned_schedule(const gconv_desc &d, const Ptrs &p) {
    std::lock_guard<std::mutex> lock(g_tuned_mutex);
    if (g_tuned.empty()) return GCONV_SCHED_AUTO;
    auto it = g_tuned.find(tune_key(d, p));
    return it == g_tuned.end() ? GCONV_SCHED_AUTO : it->second;
}

static gconv_status plan_with(const gconv_desc &d, const Ptrs &p, int32_t req, Plan *out);

static gconv_status plan_call(const gconv_desc &d, const Ptrs &p, Plan *out) {
    int32_t req = requested_schedule(d);
    if (req == GCONV_SCHED_AUTO) {
        // A schedule timed for this shape wins while it still takes the call.
        const int32_t tuned = tuned_schedule(d, p);
        if (tuned != GCONV_SCHED_AUTO && plan_with(d, p, tuned, out) == GCONV_OK) return GCONV_OK;
    }
    return plan_with(d, p, req, out);
}

static gconv_status plan_with(const gconv_desc &d, const Ptrs &p, int32_t req, Plan *out) {
    if (d.transposed) {
        gconv_desc f;
        Ptrs q;
        if (flipped_forward(d, p, &f, &q)) {
            int32_t s;
            if (select_for(f, q, req, &s) == GCONV_OK) {
                *out = Plan{f, q, s};
                return GCONV_OK;
            }
        }
    }
    int32_t s;
    gconv_status st = select_for(d, p, req, &s);
    if (st != GCONV_OK) return st;
    *out = Plan{d, p, s};
    return GCONV_OK;
}

gconv_status conv_select_schedule(const gconv_desc *d, const void *x, const void *w,
                                  const void *bias, const void *y, int32_t *schedule) {
    if (!schedule) return GCONV_ERR_NULL;
    gconv_status st = check_call(d, x, w, bias, (void *)y);
    if (st != GCONV_OK) return st;
    Plan pl;
    st = plan_call(*d, Ptrs{x, w, bias, (void *)y}, &pl);
    if (st != GCONV_OK) return st;
    *schedule = pl.schedule;
    return GCONV_OK;
}

// A CUDA error check after the launches.
static gconv_status after_launch(cudaError_t e, int launches) {
    g_launches.fetch_add((uint64_t)launches, std::memory_order_relaxed);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        t_last_cuda_error = (int32_t)e;
        return GCONV_ERR_CUDA;
    }
    return GCONV_OK;
}

static gconv_status run(const gconv_desc *d, const void *x, const void *w,
                        const void *bias, void *y, gconv_stream stream) {
    gconv_status st = check_call(d, x, w, bias, y);
    if (st != GCONV_OK) return st;
    if (empty_problem(d)) return GCONV_OK;
    Plan pl;
    st = plan_call(*d, Ptrs{x, w, bias, y}, &pl);
    if (st != GCONV_OK) return st;
    st = take_injected();
    if (st != GCONV_OK) return st;
    Params pr = make_params(pl.d);
    int launches = 0;
    cudaError_t e = kSchedules[pl.schedule]->launch(pr, pl.p, (cudaStream_t)stream, &launches);
    return after_launch(e, launches);
}

gconv_status conv_dw_forward(const gconv_desc *d, const void *x, const void *w,
                             const void *bias, void *y, gconv_stream stream) {
    if (d && d->magic == kDescMagic && d->transposed) return GCONV_ERR_KIND;
    if (d && d->magic == kDescMagic && d->Cin_g != 1) return GCONV_ERR_UNSUPPORTED;
    return run(d, x, w, bias, y, stream);
}

gconv_status conv_grouped_forward(const gconv_desc *d, const void *x, const void *w,
                                  const void *bias, void *y, gconv_stream stream) {
    if (d && d->magic == kDescMagic && d->transposed) return GCONV_ERR_KIND;
    return run(d, x, w, bias, y, stream);
}

gconv_status conv_transpose_forward(const gconv_desc *d, const void *x, const void *w,
                                    const void *bias, void *y, gconv_stream stream) {
    if (d && d->magic == kDescMagic && !d->transposed) return GCONV_ERR_KIND;
    return run(d, x, w, bias, y, stream);
}

gconv_status conv_autotune(const gconv_desc *d, const void *x, const void *w, const void *bias,
                           void *y, gconv_stream stream, int32_t reps, int32_t *schedule,
                           float *us) {
    if (reps < 1) return GCONV_ERR_SHAPE;
    gconv_status st = check_call(d, x, w, bias, y);
    if (st != GCONV_OK) return st;
    const Ptrs p{x, w, bias, y};
    if (empty_problem(d)) {
        if (schedule) *schedule = pick(*d, p);
        if (us) *us = 0.f;
        return GCONV_OK;
    }
    st = take_injected();
    if (st != GCONV_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    cudaError_t ce = cudaEventCreate(&e0);
    if (ce == cudaSuccess) ce = cudaEventCreate(&e1);
    int32_t best = GCONV_SCHED_AUTO;
    float best_ms = 0.f;
    for (int32_t sch = 0; sch < GCONV_SCHED_COUNT && ce == cudaSuccess; ++sch) {
        Plan pl;
        if (plan_with(*d, p, sch, &pl) != GCONV_OK || pl.schedule != sch) continue;
        const Params pr = make_params(pl.d);
        int launches = 0;
        ce = kSchedules[sch]->launch(pr, pl.p, s, &launches);   // warm-up
        g_launches.fetch_add((uint64_t)launches, std::memory_order_relaxed);
        if (ce == cudaSuccess) ce = cudaEventRecord(e0, s);
        for (int32_t r = 0; r < reps && ce == cudaSuccess; ++r) {
            ce = kSchedules[sch]->launch(pr, pl.p, s, &launches);
            g_launches.fetch_add((uint64_t)launches, std::memory_order_relaxed);
        }
        if (ce == cudaSuccess) ce = cudaEventRecord(e1, s);
        if (ce == cudaSuccess) ce = cudaEventSynchronize(e1);
        float ms = 0.f;
        if (ce == cudaSuccess) ce = cudaEventElapsedTime(&ms, e0, e1);
        if (ce == cudaSuccess && (best == GCONV_SCHED_AUTO || ms < best_ms)) {
            best = sch;
            best_ms = ms;
        }
    }
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    if (ce != cudaSuccess) return after_launch(ce, 0);
    if (best == GCONV_SCHED_AUTO) return GCONV_ERR_SCHEDULE;   // nothing takes the call
    {
        std::lock_guard<std::mutex> lock(g_tuned_mutex);
        g_tuned[tune_key(*d, p)] = best;
    }
    if (schedule) *schedule = best;
    if (us) *us = best_ms * 1000.f / (float)reps;
    // The last schedule timed wrote y; run the chosen one last so y holds
    // its result.
    Plan pl;
    st = plan_with(*d, p, best, &pl);
    if (st != GCONV_OK) return st;
    int launches = 0;
    ce = kSchedules[best]->launch(make_params(pl.d), pl.p, s, &launches);
    return after_launch(ce, launches);
}

void conv_autotune_clear(void) {
    std::lock_guard<std::mutex> lock(g_tuned_mutex);
    g_tuned.clear();
}

// The transposed convolution that computes dx for a forward desc: input gy
// [N, C_out, OH, OW] in y's layout, weight = the forward weight read as
// [C_in_t = C_out, Cout_g_t = Cin_g, KH, KW], crop pad_before before and
// whatever sizes the output back to H x W after (or output_padding when
// the output must grow).
static gconv_desc backward_input_desc(const gconv_desc &d) {
    gconv_desc t = d;
    t.transposed = 1;
    t.has_bias = 0;
    t.b_stride = 0;
    t.C_in = d.C_out; t.H = d.OH; t.W = d.OW;
    t.C_out = d.C_in; t.OH = d.H; t.OW = d.W;
    t.Cin_g = d.Cout_g; t.Cout_g = d.Cin_g;
    for (int i = 0; i < 4; ++i) t.x_strides[i] = d.y_strides[i];
    dense_strides(d.layout, d.N, d.C_in, d.H, d.W, t.y_strides);
    const int64_t in[2] = {d.H, d.W}, out[2] = {d.OH, d.OW}, k[2] = {d.KH, d.KW};
    for (int i = 0; i < 2; ++i) {
        const int64_t full = (out[i] - 1) * d.stride[i] + (int64_t)d.dilation[i] * (k[i] - 1) + 1;
        const int64_t r = in[i] + d.pad_before[i] - full;
        t.pad_after[i] = r < 0 ? (int32_t)-r : 0;
        t.output_padding[i] = r > 0 ? (int32_t)r : 0;
    }
    t.x_dense = 1;
    t.schedule = d.schedule;
    return t;
}

gconv_status conv_backward_input(const gconv_desc *d, const void *gy, const void *w,
                                 void *dx, gconv_stream stream) {
    if (!d) return GCONV_ERR_NULL;
    if (d->magic != kDescMagic) return GCONV_ERR_INTERNAL;
    if (d->transposed) return GCONV_ERR_KIND;
    if (d->N == 0 || d->C_in == 0 || d->H == 0 || d->W == 0) return GCONV_OK;
    if (!dx) return GCONV_ERR_NULL;
    if (d->C_out == 0) {
        // No output channel reads x: the gradient is zero.
        gconv_status st = take_injected();
        if (st != GCONV_OK) return st;
        const size_t bytes = (size_t)(d->N * d->C_in * d->H * d->W) * dtype_size(d->dtype);
        return after_launch(cudaMemsetAsync(dx, 0, bytes, (cudaStream_t)stream), 1);
    }
    if (!gy || !w) return GCONV_ERR_NULL;
    const gconv_desc t = backward_input_desc(*d);
    return run(&t, gy, w, nullptr, dx, stream);
}

gconv_status conv_backward_weight_workspace_size(const gconv_desc *d, uint64_t *bytes) {
    if (!d || !bytes) return GCONV_ERR_NULL;
    if (d->magic != kDescMagic) return GCONV_ERR_INTERNAL;
    if (d->transposed) return GCONV_ERR_KIND;
    *bytes = wgrad_workspace_bytes(make_params(*d));
    return GCONV_OK;
}

gconv_status conv_backward_weight(const gconv_desc *d, const void *x, const void *gy,
                                  void *dw, void *db, void *workspace,
                                  uint64_t workspace_bytes, gconv_stream stream) {
    if (!d) return GCONV_ERR_NULL;
    if (d->magic != kDescMagic) return GCONV_ERR_INTERNAL;
    if (d->transposed) return GCONV_ERR_KIND;
    if (d->C_out == 0) return GCONV_OK;
    if (!dw) return GCONV_ERR_NULL;
    const bool has_pixels = d->N > 0 && d->OH > 0 && d->OW > 0;
    if (has_pixels && (!x || !gy)) return GCONV_ERR_NULL;
    const Params pr = make_params(*d);
    const uint64_t need = wgrad_workspace_bytes(pr);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 16))
        return GCONV_ERR_WORKSPACE;
    gconv_status st = take_injected();
    if (st != GCONV_OK) return st;
    int launches = 0;
    cudaError_t e = wgrad_launch(pr, x, gy, dw, db, workspace, (cudaStream_t)stream, &launches);
    return after_launch(e, launches);
}

gconv_status conv_force_schedule(int32_t schedule) {
    if (schedule < GCONV_SCHED_AUTO || schedule >= GCONV_SCHED_COUNT) return GCONV_ERR_SCHEDULE;
    g_forced.store(schedule);
    return GCONV_OK;
}

const char *conv_schedule_name(int32_t schedule) {
    if (schedule == GCONV_SCHED_AUTO) return "auto";
    if (schedule < 0 || schedule >= GCONV_SCHED_COUNT) return "unknown";
    return kSchedules[schedule]->name;
}

const char *conv_strerror(gconv_status s) {
    switch (s) {
    case GCONV_OK: return "ok";
    case GCONV_ERR_NULL: return "required pointer is NULL (or bias presence does not match the desc)";
    case GCONV_ERR_RANK: return "x must be rank 3 or 4, w rank 4 and bias rank 1";
    case GCONV_ERR_DTYPE: return "unknown dtype";
    case GCONV_ERR_SHAPE: return "channel, group, weight, bias or stride mismatch";
    case GCONV_ERR_UNSUPPORTED: return "outside the envelope (dilation >= 1, kernel <= 9x9, <= 8 input channels per group)";
    case GCONV_ERR_PADDING: return "negative padding or window larger than the padded input";
    case GCONV_ERR_ALIGN: return "forced schedule needs more pointer alignment";
    case GCONV_ERR_CUDA: return "CUDA launch failed";
    case GCONV_ERR_INTERNAL: return "descriptor not produced by conv_bind, or size overflow";
    case GCONV_ERR_LAYOUT: return "x is neither NCHW- nor channels-last-ordered";
    case GCONV_ERR_SCHEDULE: return "forced schedule does not support this convolution";
    case GCONV_ERR_KIND: return "descriptor of another operation (forward vs transposed)";
    case GCONV_ERR_WORKSPACE: return "workspace missing, too small or not 16-byte aligned";
    case GCONV_ERR_SCRATCH_LIMIT: return "needs more scratch than the library's fixed device buffer holds";
    }
    return "unknown status";
}

void conv_test_inject_launch_error(int32_t cuda_error) { g_inject.store(cuda_error); }

int32_t conv_last_cuda_error(void) { return t_last_cuda_error; }

uint64_t conv_launch_count(void) { return g_launches.load(); }

int32_t conv_version(void) { return 200; }

}  // extern "C"
