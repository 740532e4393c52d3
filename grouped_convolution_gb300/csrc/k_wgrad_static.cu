// k_wgrad_static.cu -- conv_backward_weight_noalloc: the weight / bias
// gradient with its scratch in a fixed device buffer that the library owns,
// for callers that cannot hand it a workspace.
//
// Who needs it: code that runs inside a host framework which owns every
// device allocation (only the framework's pool may be used, and this library
// has no handle to it), and code on a fixed memory budget that forbids any
// allocation after start-up.  Such a caller can pass inputs and outputs it
// was given, but cannot call cudaMalloc for a workspace, and a cudaMalloc
// may also synchronise the device in the middle of its stream work.
//
// The buffer is a file-scope __device__ array of kWgradStaticBytes: every
// GPU that loads the library holds it until the process exits.  Host code
// cannot pass the array's name to a kernel (in host code it names a host-side
// stand-in, not device memory), so the device address is looked up with
// cudaGetSymbolAddress on the first call made in a context and cached with
// that context.  A call made in another context (after a cudaDeviceReset
// created a new primary context, which may place the array elsewhere)
// looks it up again.  The first call in a context should come before any
// stream capture begins.
// Nothing here allocates: no cudaMalloc, no cudaFree, no allocating library
// routine.
//
// Every call shares the one buffer and leaves its contents behind.  The
// partial pass writes every entry it later reads, so nothing has to start at
// zero; but two calls whose kernels overlap on the GPU (different streams
// without ordering, or two host threads on different streams) race on the
// buffer and give wrong results.  Order such calls on one stream.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <mutex>

#include "gconv_internal.h"

namespace gconv {
namespace {

constexpr uint64_t kWgradStaticBytes = 8ull << 20;   // 8 MiB per device

__device__ __align__(256) unsigned char g_wgrad_scratch[kWgradStaticBytes];

constexpr int kMaxDevices = 64;

// cuCtxGetCurrent, resolved once through the runtime (the library does not
// link the driver library).
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(f);
    });
    return fn;
}

struct ScratchEntry {
    void *ctx = nullptr;    // the context the address was looked up in
    void *addr = nullptr;
};
ScratchEntry g_scratch[kMaxDevices];
std::mutex g_scratch_mutex;

// The buffer's device address in the current context.
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    CUcontext ctx = nullptr;
    CtxGetCurrentFn fn = ctx_get_current();
    const bool have_ctx = fn && fn(&ctx) == CUDA_SUCCESS && ctx != nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchEntry &en = g_scratch[dev];
    if (have_ctx && en.addr && en.ctx == (void *)ctx) {
        *out = en.addr;
        return cudaSuccess;
    }
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_wgrad_scratch);
    if (e != cudaSuccess) return e;
    if (have_ctx) {
        en.ctx = (void *)ctx;
        en.addr = p;
    }
    *out = p;
    return cudaSuccess;
}

}  // namespace
}  // namespace gconv

using namespace gconv;

extern "C" {

uint64_t conv_backward_weight_noalloc_limit(void) { return kWgradStaticBytes; }

gconv_status conv_backward_weight_noalloc(const gconv_desc *d, const void *x, const void *gy,
                                          void *dw, void *db, gconv_stream stream) {
    if (!d) return GCONV_ERR_NULL;
    if (d->magic != kDescMagic) return GCONV_ERR_INTERNAL;
    if (d->transposed) return GCONV_ERR_KIND;
    if (d->C_out == 0) return GCONV_OK;
    if (!dw) return GCONV_ERR_NULL;
    const bool has_pixels = d->N > 0 && d->OH > 0 && d->OW > 0;
    if (has_pixels && (!x || !gy)) return GCONV_ERR_NULL;
    const Params pr = make_params(*d);
    if (wgrad_workspace_bytes(pr) > kWgradStaticBytes) return GCONV_ERR_SCRATCH_LIMIT;
    const gconv_status inj = take_injected();
    if (inj != GCONV_OK) return inj;
    void *scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e == cudaSuccess) {
        int launches = 0;
        e = wgrad_launch(pr, x, gy, dw, db, scratch, (cudaStream_t)stream, &launches);
        note_launches(launches);
        if (e == cudaSuccess) e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
        note_cuda_error((int32_t)e);
        return GCONV_ERR_CUDA;
    }
    return GCONV_OK;
}

}  // extern "C"
