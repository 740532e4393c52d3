// gconv_internal.h -- shared declarations between the host library and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/gconv.h"

namespace gconv {

constexpr uint32_t kDescMagic = 0x47434f4eu;  // "GCON"

// Everything a kernel needs, by value.  Spatial and channel extents are
// checked by conv_bind to fit in int32; strides stay 64-bit.
struct Params {
    int N, C_in, H, W, C_out, G, Cin_g, Cout_g, KH, KW, OH, OW;
    int sh, sw, pbh, pbw;
    int dh, dw;      // dilation
    int transposed;  // 1: y gathers x at (o + pb - k*d) / s (weight [C_in, Cout_g, KH, KW])
    int has_bias, layout, dtype;
    int64_t xs[4];   // x strides, logical (N, C, H, W)
    int64_t ws[4];   // w strides, logical (C_out, Cin_g, KH, KW)
    int64_t bs;      // bias stride
    int64_t ys[4];   // y strides, logical (N, C_out, OH, OW)
};

struct Ptrs {
    const void *x;
    const void *w;
    const void *b;   // nullptr when there is no bias
    void *y;
};

Params make_params(const gconv_desc &d);

// One launcher per schedule.  `supports` is pure host logic (shape, layout,
// alignment); `launch` enqueues the kernel(s) and returns the launch count.
struct Schedule {
    const char *name;
    bool (*supports)(const gconv_desc &d, const Ptrs &p);
    cudaError_t (*launch)(const Params &pr, const Ptrs &p, cudaStream_t s, int *launches);
};

// Programmatic dependent launch for the library's kernels: GCONV_PDL=1 in
// the environment (read once).
bool pdl_enabled();

// Schedules, indexed by gconv_schedule.
extern const Schedule kDwFlat;
extern const Schedule kDwRow8;
extern const Schedule kDwMult;
extern const Schedule kGrpPlane;
extern const Schedule kGrpReduce;
extern const Schedule kGrpTc;
extern const Schedule kDwLine;
extern const Schedule kDwSmall;
extern const Schedule kDwTc;
extern const Schedule kDwTcl;

// The plain forward convolution of the direct-stencil envelope (dilation 1,
// not transposed): the only calls the specialised schedules take.
inline bool plain_forward(const gconv_desc &d) {
    return !d.transposed && d.dilation[0] == 1 && d.dilation[1] == 1;
}

// Bookkeeping shared by entry points outside host.cpp: the launch counter
// behind conv_launch_count and the error behind conv_last_cuda_error.
void note_launches(int launches);
void note_cuda_error(int32_t e);
// conv_test_inject_launch_error's pending value: GCONV_ERR_CUDA (recording
// the value as the last CUDA error) instead of launching, once.
gconv_status take_injected();

// grp_tc's shift form (k_tcs.cu): stride-2 grouped calls with 4 or 8
// channels per group whose chunk holds 8 or 16 output channels.
bool tcs_takes(const Params &p, const void *x);
bool tcs_supports(const gconv_desc &d, const Ptrs &q);
cudaError_t tcs_launch(const Params &p, const Ptrs &q, cudaStream_t s, int *launches);

// Backward weight pass (k_wgrad.cu): workspace bytes, and the launches.
uint64_t wgrad_workspace_bytes(const Params &p);
cudaError_t wgrad_launch(const Params &p, const void *x, const void *gy, void *dw, void *db,
                         void *workspace, cudaStream_t s, int *launches);

// Its partial pass on the dw_row8 row ring (k_wgrad_row.cu), for channels-last
// depthwise 3x3 calls at square stride 1 or 2: the workspace slices it writes
// (0 when the shape is not taken), its pointer condition, and the launch.
int wgrad_row_slices(const Params &p);
bool wgrad_row_pointers(const void *x, const void *gy);
cudaError_t wgrad_row_partial(const Params &p, const void *x, const void *gy, float *ws,
                              cudaStream_t s);

inline bool aligned(const void *p, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

inline int dtype_size(int dt) { return dt == GCONV_F32 ? 4 : 2; }

}  // namespace gconv
