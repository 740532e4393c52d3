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

#include "gconv_internal.h"

using namespace gconv;

namespace {

std::atomic<int32_t> g_forced{INT32_MIN};   // INT32_MIN: not yet read from env
std::atomic<int32_t> g_inject{0};
std::atomic<uint64_t> g_launches{0};
thread_local int32_t t_last_cuda_error = 0;

const Schedule *const kSchedules[GCONV_SCHED_COUNT] = {
    &kDwFlat, &kDwRow8, &kDwMult, &kGrpPlane, &kGrpReduce, &kGrpTc};

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

Params make_params(const gconv_desc &d) {
    Params p{};
    p.N = (int)d.N; p.C_in = (int)d.C_in; p.H = (int)d.H; p.W = (int)d.W;
    p.C_out = (int)d.C_out; p.G = (int)d.groups; p.Cin_g = (int)d.Cin_g;
    p.Cout_g = (int)d.Cout_g; p.KH = (int)d.KH; p.KW = (int)d.KW;
    p.OH = (int)d.OH; p.OW = (int)d.OW;
    p.sh = d.stride[0]; p.sw = d.stride[1];
    p.pbh = d.pad_before[0]; p.pbw = d.pad_before[1];
    p.has_bias = d.has_bias; p.layout = d.layout; p.dtype = d.dtype;
    for (int i = 0; i < 4; ++i) {
        p.xs[i] = d.x_strides[i]; p.ws[i] = d.w_strides[i]; p.ys[i] = d.y_strides[i];
    }
    p.bs = d.b_stride;
    return p;
}

}  // namespace gconv

extern "C" {

gconv_status conv_bind(const gconv_tensor *x, const gconv_tensor *w,
                       const gconv_tensor *bias, int32_t dtype,
                       const int32_t stride[2], const int32_t padding_before[2],
                       const int32_t padding_after[2], const int32_t dilation[2],
                       int64_t groups, gconv_desc *out) {
    if (!x || !w || !out) return GCONV_ERR_NULL;
    gconv_desc d;
    memset(&d, 0, sizeof(d));
    if (dtype != GCONV_F32 && dtype != GCONV_F16 && dtype != GCONV_BF16)
        return GCONV_ERR_DTYPE;
    if (x->rank != 3 && x->rank != 4) return GCONV_ERR_RANK;
    if (w->rank != 4) return GCONV_ERR_RANK;
    if (bias && bias->rank != 1) return GCONV_ERR_RANK;

    // Canonical x geometry [N, C, H, W]; rank 3 is one image.
    int64_t xs[4], xst[4];
    if (x->rank == 3) {
        xs[0] = 1; xst[0] = 0;
        for (int i = 0; i < 3; ++i) { xs[i + 1] = x->sizes[i]; xst[i + 1] = x->strides[i]; }
        d.unbatched = 1;
    } else {
        for (int i = 0; i < 4; ++i) { xs[i] = x->sizes[i]; xst[i] = x->strides[i]; }
    }
    for (int i = 0; i < 4; ++i) {
        if (xs[i] < 0 || w->sizes[i] < 0) return GCONV_ERR_SHAPE;
        if (!fits_i32(xs[i]) || !fits_i32(w->sizes[i])) return GCONV_ERR_UNSUPPORTED;
        if (xst[i] < 0 || w->strides[i] < 0) return GCONV_ERR_LAYOUT;
    }
    const int64_t N = xs[0], C_in = xs[1], H = xs[2], W = xs[3];
    const int64_t C_out = w->sizes[0], Cin_g = w->sizes[1], KH = w->sizes[2], KW = w->sizes[3];

    // Scalars: NULL pointers take the canonical defaults.
    int32_t st[2] = {1, 1}, pb[2] = {0, 0}, pa[2] = {0, 0}, dil[2] = {1, 1};
    if (stride) { st[0] = stride[0]; st[1] = stride[1]; }
    if (padding_before) { pb[0] = padding_before[0]; pb[1] = padding_before[1]; }
    if (padding_after) { pa[0] = padding_after[0]; pa[1] = padding_after[1]; }
    if (dilation) { dil[0] = dilation[0]; dil[1] = dilation[1]; }

    // Group shape: C_in == Cin_g * groups (torch/_inductor/kernel/conv.py,
    // convolution: in_chan * groups == C_in), groups divides C_out.
    if (groups < 1) return GCONV_ERR_SHAPE;
    if (Cin_g < 1 || Cin_g * groups != C_in) return GCONV_ERR_SHAPE;
    if (C_out % groups != 0) return GCONV_ERR_SHAPE;
    if (bias) {
        if (bias->sizes[0] != C_out) return GCONV_ERR_SHAPE;
        if (bias->strides[0] < 0) return GCONV_ERR_LAYOUT;
    }
    if (st[0] < 1 || st[1] < 1) return GCONV_ERR_SHAPE;

    // The direct-stencil envelope.
    if (dil[0] != 1 || dil[1] != 1) return GCONV_ERR_UNSUPPORTED;
    if (KH < 1 || KH > 9 || KW < 1 || KW > 9) return GCONV_ERR_UNSUPPORTED;
    if (Cin_g > 8) return GCONV_ERR_UNSUPPORTED;

    if (pb[0] < 0 || pb[1] < 0 || pa[0] < 0 || pa[1] < 0) return GCONV_ERR_PADDING;
    const int64_t Hp = H + pb[0] + pa[0], Wp = W + pb[1] + pa[1];
    if (Hp < KH || Wp < KW) return GCONV_ERR_PADDING;
    const int64_t OH = (Hp - KH) / st[0] + 1, OW = (Wp - KW) / st[1] + 1;
    if (!fits_i32(OH) || !fits_i32(OW)) return GCONV_ERR_UNSUPPORTED;

    // Layout of x: NCHW-ordered or channels-last-ordered; NCHW on a tie.
    static const int kNCHW[4] = {0, 1, 2, 3}, kNHWC[4] = {0, 2, 3, 1};
    bool dense_nchw = false, dense_nhwc = false;
    if (ordered(xs, xst, kNCHW, &dense_nchw)) {
        d.layout = GCONV_LAYOUT_NCHW;
        d.x_dense = dense_nchw;
    } else if (ordered(xs, xst, kNHWC, &dense_nhwc)) {
        d.layout = GCONV_LAYOUT_NHWC;
        d.x_dense = dense_nhwc;
    } else {
        return GCONV_ERR_LAYOUT;
    }

    // Size products must stay far from int64 overflow.
    const double big = 4.0e18;
    if ((double)N * C_out * OH * OW > big || (double)N * C_in * H * W > big)
        return GCONV_ERR_UNSUPPORTED;

    d.dtype = dtype;
    d.has_bias = bias != nullptr;
    d.schedule = GCONV_SCHED_AUTO;
    d.N = N; d.C_in = C_in; d.H = H; d.W = W;
    d.C_out = C_out; d.groups = groups; d.Cin_g = Cin_g; d.Cout_g = C_out / groups;
    d.KH = KH; d.KW = KW; d.OH = OH; d.OW = OW;
    d.stride[0] = st[0]; d.stride[1] = st[1];
    d.pad_before[0] = pb[0]; d.pad_before[1] = pb[1];
    d.pad_after[0] = pa[0]; d.pad_after[1] = pa[1];
    for (int i = 0; i < 4; ++i) { d.x_strides[i] = xst[i]; d.w_strides[i] = w->strides[i]; }
    d.b_stride = bias ? bias->strides[0] : 0;
    if (d.layout == GCONV_LAYOUT_NCHW) {
        d.y_strides[3] = 1;
        d.y_strides[2] = OW;
        d.y_strides[1] = OH * OW;
        d.y_strides[0] = C_out * OH * OW;
    } else {
        d.y_strides[1] = 1;
        d.y_strides[3] = C_out;
        d.y_strides[2] = OW * C_out;
        d.y_strides[0] = OH * OW * C_out;
    }
    d.magic = kDescMagic;
    *out = d;
    return GCONV_OK;
}

gconv_status out_shape_and_stride(const gconv_desc *d, int32_t *rank,
                                  int64_t sizes[4], int64_t strides[4]) {
    if (!d || !rank || !sizes || !strides) return GCONV_ERR_NULL;
    if (d->magic != kDescMagic) return GCONV_ERR_INTERNAL;
    const int64_t s4[4] = {d->N, d->C_out, d->OH, d->OW};
    if (d->unbatched) {
        *rank = 3;
        for (int i = 0; i < 3; ++i) { sizes[i] = s4[i + 1]; strides[i] = d->y_strides[i + 1]; }
        sizes[3] = 0; strides[3] = 0;
    } else {
        *rank = 4;
        for (int i = 0; i < 4; ++i) { sizes[i] = s4[i]; strides[i] = d->y_strides[i]; }
    }
    return GCONV_OK;
}

// The per-shape picker.  Specialised schedules win where they apply; the
// fallback schedule dw_flat takes everything else.  Grouped calls the
// tensor cores can take (4 or 8 channels per group, channels-last 16-bit)
// run there.  Other calls with too few outputs to give every thread of the
// GPU its own (fewer than 152 SMs x 512) and a long tap loop split the taps
// across lanes instead.
static int32_t pick(const gconv_desc &d, const Ptrs &p) {
    const bool dw = d.Cin_g == 1;
    if (dw && d.Cout_g == 1 && kDwRow8.supports(d, p)) return GCONV_SCHED_DW_ROW8;
    if (dw && kDwMult.supports(d, p)) return GCONV_SCHED_DW_MULT;
    if (!dw && kGrpTc.supports(d, p)) return GCONV_SCHED_GRP_TC;
    const double outputs = (double)d.N * d.C_out * d.OH * d.OW;
    const int64_t taps = d.Cin_g * d.KH * d.KW;
    if (outputs < 152.0 * 512 && taps >= 32) return GCONV_SCHED_GRP_REDUCE;
    if (kGrpPlane.supports(d, p)) return GCONV_SCHED_GRP_PLANE;
    return GCONV_SCHED_DW_FLAT;
}

static gconv_status select_impl(const gconv_desc *d, const Ptrs &p, int32_t *out) {
    int32_t s = d->schedule;
    if (s == GCONV_SCHED_AUTO) s = forced_schedule();
    if (s == GCONV_SCHED_AUTO) {
        *out = pick(*d, p);
        return GCONV_OK;
    }
    if (s < 0 || s >= GCONV_SCHED_COUNT) return GCONV_ERR_SCHEDULE;
    if (!kSchedules[s]->supports(*d, p)) {
        // Distinguish "this shape never runs here" from "these pointers are
        // not aligned enough": retry with ideally aligned pointers.
        Ptrs ideal{(const void *)(uintptr_t)4096, (const void *)(uintptr_t)4096,
                   p.b ? (const void *)(uintptr_t)4096 : nullptr, (void *)(uintptr_t)4096};
        return kSchedules[s]->supports(*d, ideal) ? GCONV_ERR_ALIGN : GCONV_ERR_SCHEDULE;
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

gconv_status conv_select_schedule(const gconv_desc *d, const void *x, const void *w,
                                  const void *bias, const void *y, int32_t *schedule) {
    if (!schedule) return GCONV_ERR_NULL;
    gconv_status st = check_call(d, x, w, bias, (void *)y);
    if (st != GCONV_OK) return st;
    Ptrs p{x, w, bias, (void *)y};
    return select_impl(d, p, schedule);
}

static gconv_status forward(const gconv_desc *d, const void *x, const void *w,
                            const void *bias, void *y, gconv_stream stream) {
    gconv_status st = check_call(d, x, w, bias, y);
    if (st != GCONV_OK) return st;
    if (empty_problem(d)) return GCONV_OK;
    Ptrs p{x, w, bias, y};
    int32_t s;
    st = select_impl(d, p, &s);
    if (st != GCONV_OK) return st;
    int32_t inj = g_inject.exchange(0);
    if (inj != 0) {
        t_last_cuda_error = inj;
        return GCONV_ERR_CUDA;
    }
    Params pr = make_params(*d);
    int launches = 0;
    cudaError_t e = kSchedules[s]->launch(pr, p, (cudaStream_t)stream, &launches);
    g_launches.fetch_add((uint64_t)launches, std::memory_order_relaxed);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        t_last_cuda_error = (int32_t)e;
        return GCONV_ERR_CUDA;
    }
    return GCONV_OK;
}

gconv_status conv_dw_forward(const gconv_desc *d, const void *x, const void *w,
                             const void *bias, void *y, gconv_stream stream) {
    if (d && d->magic == kDescMagic && d->Cin_g != 1) return GCONV_ERR_UNSUPPORTED;
    return forward(d, x, w, bias, y, stream);
}

gconv_status conv_grouped_forward(const gconv_desc *d, const void *x, const void *w,
                                  const void *bias, void *y, gconv_stream stream) {
    return forward(d, x, w, bias, y, stream);
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
    case GCONV_ERR_UNSUPPORTED: return "outside the direct-stencil envelope (dilation 1, kernel <= 9x9, <= 8 input channels per group)";
    case GCONV_ERR_PADDING: return "negative padding or window larger than the padded input";
    case GCONV_ERR_ALIGN: return "forced schedule needs more pointer alignment";
    case GCONV_ERR_CUDA: return "CUDA launch failed";
    case GCONV_ERR_INTERNAL: return "descriptor not produced by conv_bind, or size overflow";
    case GCONV_ERR_LAYOUT: return "x is neither NCHW- nor channels-last-ordered";
    case GCONV_ERR_SCHEDULE: return "forced schedule does not support this convolution";
    }
    return "unknown status";
}

void conv_test_inject_launch_error(int32_t cuda_error) { g_inject.store(cuda_error); }

int32_t conv_last_cuda_error(void) { return t_last_cuda_error; }

uint64_t conv_launch_count(void) { return g_launches.load(); }

int32_t conv_version(void) { return 100; }

}  // extern "C"
