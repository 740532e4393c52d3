// device_common.cuh -- element conversions and small helpers shared by the
// kernels.  All arithmetic is fp32; inputs are widened exactly and the result
// is rounded once, to nearest even, by the hardware conversion.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace gconv {

template <typename T> struct Elem;

template <> struct Elem<float> {
    static __device__ __forceinline__ float load(const float *p) { return __ldg(p); }
    static __device__ __forceinline__ float to_f32(float v) { return v; }
    static __device__ __forceinline__ float from_f32(float v) { return v; }
};

template <> struct Elem<__half> {
    static __device__ __forceinline__ float load(const __half *p) { return __half2float(__ldg(p)); }
    static __device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }
    static __device__ __forceinline__ __half from_f32(float v) { return __float2half_rn(v); }
};

template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float load(const __nv_bfloat16 *p) {
        return __bfloat162float(__ldg(p));
    }
    static __device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
    static __device__ __forceinline__ __nv_bfloat16 from_f32(float v) { return __float2bfloat16_rn(v); }
};

// Widen the two 16-bit values packed in a 32-bit word (low half first).
__device__ __forceinline__ float2 unpack2(uint32_t v, __nv_bfloat16 *) {
    // bf16 -> fp32 is exact: the 16 bits become the top half of the word.
    return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}
__device__ __forceinline__ float2 unpack2(uint32_t v, __half *) {
    __half2 h = *reinterpret_cast<__half2 *>(&v);
    return __half22float2(h);
}

// Round two fp32 values to one packed 32-bit word (low half first).
__device__ __forceinline__ uint32_t pack2(float a, float b, __nv_bfloat16 *) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint32_t pack2(float a, float b, __half *) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

template <typename T>
__device__ __forceinline__ float load_f32(const T *p) { return Elem<T>::load(p); }

// Division of 32-bit unsigned n by a divisor d fixed for a launch, by a
// multiply-high and shifts (T. Granlund and P. L. Montgomery, "Division by
// invariant integers using multiplication", PLDI 1994, section 4: with
// l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1,
// q = (t + ((n - t) >> 1)) >> (l - 1) where t = mulhi(m, n), for l >= 1;
// q = n for d = 1).  A runtime integer division costs tens of
// instructions; this costs four.  Built on the host, used on the device.
struct FastDiv {
    uint32_t d, m, l;
    FastDiv() : d(1), m(0), l(0) {}
    explicit FastDiv(uint32_t dd) : d(dd ? dd : 1), m(0), l(0) {
        while ((1ull << l) < d) ++l;
        if (l > 0) m = (uint32_t)(((1ull << 32) * ((1ull << l) - d)) / d + 1);
    }
    __host__ __device__ __forceinline__ uint32_t div(uint32_t n) const {
        if (l == 0) return n;
#ifdef __CUDA_ARCH__
        const uint32_t t = __umulhi(m, n);
#else
        const uint32_t t = (uint32_t)(((uint64_t)m * n) >> 32);
#endif
        return (t + ((n - t) >> 1)) >> (l - 1);
    }
    // n = q*d + r
    __host__ __device__ __forceinline__ void divmod(uint32_t n, uint32_t &q, uint32_t &r) const {
        q = div(n);
        r = n - q * d;
    }
};

// The input index that output index o reads at tap k along one dim, or -1
// when the tap falls outside the input.  Forward: o*s - pb + k*d (the conv.py
// LOOP_BODY_2D rule with dilation).  Transposed (executorch PR #25091,
// description, second paragraph): (o + pb - k*d) / s when that is a whole
// number.
template <bool TR>
__device__ __forceinline__ int tap_input(int o, int k, int s, int pb, int d, int n_in) {
    if constexpr (!TR) {
        const int i = o * s - pb + k * d;
        return (i >= 0 && i < n_in) ? i : -1;
    } else {
        const int t = o + pb - k * d;
        if (t < 0) return -1;
        const int i = t / s;
        return (i * s == t && i < n_in) ? i : -1;
    }
}

template <typename T>
__device__ __forceinline__ T from_f32(float v) { return Elem<T>::from_f32(v); }

}  // namespace gconv

// Dispatch a templated launcher on the runtime dtype code.
#define GCONV_DISPATCH_DTYPE(dt, T, ...)                            \
    [&]() -> cudaError_t {                                          \
        switch (dt) {                                               \
        case GCONV_F32: { using T = float; return __VA_ARGS__(); }  \
        case GCONV_F16: { using T = __half; return __VA_ARGS__(); } \
        case GCONV_BF16: { using T = __nv_bfloat16; return __VA_ARGS__(); } \
        }                                                           \
        return cudaErrorInvalidValue;                               \
    }()
