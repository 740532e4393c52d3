// k_probe.cu -- conv_probe_fma_rate: a launch of independent fp32 FMA chains
// that keeps every FP32 lane of every SM busy, so a caller can time it and
// state the chip's measured FMA rate, the denominator of the FMA-bound
// convolutions' roofline (a depthwise stencil does one fp32 FMA per tap and
// output, on the same FP32 pipe).
#include "gconv_internal.h"

namespace {

constexpr int kProbeThreads = 256;
constexpr int kProbeChains = 8;    // independent accumulators per thread
constexpr int kProbeUnroll = 16;   // FMAs per chain per loop trip

__global__ void __launch_bounds__(kProbeThreads)
fma_probe_kernel(float *out, int trips, float a, float c) {
    float r[kProbeChains];
#pragma unroll
    for (int i = 0; i < kProbeChains; ++i) r[i] = (float)(threadIdx.x + i) * 1e-3f;
    for (int t = 0; t < trips; ++t) {
#pragma unroll
        for (int u = 0; u < kProbeUnroll; ++u) {
#pragma unroll
            for (int i = 0; i < kProbeChains; ++i) r[i] = fmaf(r[i], a, c);
        }
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kProbeChains; ++i) s += r[i];
    // A store the compiler cannot prove dead; with a = 1 - 2^-20 and c = 0 the
    // chains decay toward zero and never reach the sentinel.
    if (s == 12345.f) out[blockIdx.x] = s;
}

}  // namespace

extern "C" {

gconv_status conv_probe_fma_rate(int32_t trips, float *sink, gconv_stream stream,
                                 uint64_t *fmas) {
    if (!sink || !fmas) return GCONV_ERR_NULL;
    if (trips < 1) return GCONV_ERR_SHAPE;
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fma_probe_kernel,
                                                          kProbeThreads, 0);
    if (e != cudaSuccess) {
        gconv::note_cuda_error((int32_t)e);
        return GCONV_ERR_CUDA;
    }
    const int blocks = sms * (per_sm > 0 ? per_sm : 1);
    fma_probe_kernel<<<blocks, kProbeThreads, 0, (cudaStream_t)stream>>>(
        sink, trips, 1.0f - 9.5367431640625e-7f, 0.0f);
    e = cudaGetLastError();
    gconv::note_launches(1);
    if (e != cudaSuccess) {
        gconv::note_cuda_error((int32_t)e);
        return GCONV_ERR_CUDA;
    }
    *fmas = (uint64_t)blocks * kProbeThreads * kProbeChains * kProbeUnroll * (uint64_t)trips;
    return GCONV_OK;
}

}  // extern "C"
