// stencil_math.cuh -- vectors, widening and the multiply-accumulate step of
// the stencils.
//
// fp32 accumulation throughout.  16-bit inputs are widened once per load
// (bf16 -> fp32 is a 16-bit shift, fp16 -> fp32 the hardware conversion),
// then every product is an fp32 FMA.  Values travel as channel pairs
// (float2) because two 16-bit channels share one 32-bit word.  Measured on
// GB300: the packed fma.rn.f32x2 issues as one instruction but runs only on
// one of the two FMA pipes, while scalar FMAs use both; which is faster
// depends on the kernel (issue slots vs latency), so both forms exist.
#pragma once

#include "device_common.cuh"

namespace gconv {

// A vector of VEC elements of T held as 32-bit words.
template <typename T, int VEC> struct Vec {
    static_assert(VEC * sizeof(T) >= 4, "a vector holds at least one 32-bit word");
    static constexpr int kBytes = VEC * (int)sizeof(T);
    static constexpr int kWords = kBytes / 4;
    uint32_t w[kWords];
};

template <int BYTES> struct VecIO;
template <> struct VecIO<4> {
    template <typename V> static __device__ __forceinline__ void load(V &v, const void *p) {
        v.w[0] = __ldg(reinterpret_cast<const unsigned int *>(p));
    }
    template <typename V> static __device__ __forceinline__ void load_shared(V &v, const void *p) {
        v.w[0] = *reinterpret_cast<const unsigned int *>(p);
    }
    template <typename V> static __device__ __forceinline__ void store(void *p, const V &v) {
        *reinterpret_cast<unsigned int *>(p) = v.w[0];
    }
};
template <> struct VecIO<8> {
    template <typename V> static __device__ __forceinline__ void load(V &v, const void *p) {
        uint2 t = __ldg(reinterpret_cast<const uint2 *>(p));
        v.w[0] = t.x; v.w[1] = t.y;
    }
    template <typename V> static __device__ __forceinline__ void load_shared(V &v, const void *p) {
        uint2 t = *reinterpret_cast<const uint2 *>(p);
        v.w[0] = t.x; v.w[1] = t.y;
    }
    template <typename V> static __device__ __forceinline__ void store(void *p, const V &v) {
        *reinterpret_cast<uint2 *>(p) = make_uint2(v.w[0], v.w[1]);
    }
};
template <> struct VecIO<16> {
    template <typename V> static __device__ __forceinline__ void load(V &v, const void *p) {
        uint4 t = __ldg(reinterpret_cast<const uint4 *>(p));
        v.w[0] = t.x; v.w[1] = t.y; v.w[2] = t.z; v.w[3] = t.w;
    }
    template <typename V> static __device__ __forceinline__ void load_shared(V &v, const void *p) {
        uint4 t = *reinterpret_cast<const uint4 *>(p);
        v.w[0] = t.x; v.w[1] = t.y; v.w[2] = t.z; v.w[3] = t.w;
    }
    template <typename V> static __device__ __forceinline__ void store(void *p, const V &v) {
        *reinterpret_cast<uint4 *>(p) = make_uint4(v.w[0], v.w[1], v.w[2], v.w[3]);
    }
};

// Widen a vector of VEC (even) elements into VEC/2 fp32 channel pairs.
template <typename T, int VEC>
__device__ __forceinline__ void widen(const Vec<T, VEC> &v, float2 (&f)[VEC / 2]) {
    static_assert(VEC % 2 == 0, "channel pairs");
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int k = 0; k < VEC / 2; ++k)
            f[k] = make_float2(__uint_as_float(v.w[2 * k]), __uint_as_float(v.w[2 * k + 1]));
    } else {
#pragma unroll
        for (int k = 0; k < VEC / 2; ++k) f[k] = unpack2(v.w[k], (T *)nullptr);
    }
}

template <typename T, int VEC>
__device__ __forceinline__ void zero(float2 (&f)[VEC / 2]) {
#pragma unroll
    for (int k = 0; k < VEC / 2; ++k) f[k] = make_float2(0.f, 0.f);
}

// acc += w * x on one channel pair (two scalar round-to-nearest FMAs).
__device__ __forceinline__ void fma2(float2 &acc, float2 w, float2 x) {
    acc.x = fmaf(w.x, x.x, acc.x);
    acc.y = fmaf(w.y, x.y, acc.y);
}

// The same with one packed fma.rn.f32x2 (both lanes round to nearest).
__device__ __forceinline__ void fma2_packed(float2 &acc, float2 w, float2 x) {
    acc = __ffma2_rn(w, x, acc);
}

// Round VEC fp32 values (as pairs) to T and pack them.
template <typename T, int VEC>
__device__ __forceinline__ Vec<T, VEC> pack_pairs(const float2 (&a)[VEC / 2]) {
    Vec<T, VEC> r;
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int k = 0; k < VEC / 2; ++k) {
            r.w[2 * k] = __float_as_uint(a[k].x);
            r.w[2 * k + 1] = __float_as_uint(a[k].y);
        }
    } else {
#pragma unroll
        for (int k = 0; k < VEC / 2; ++k) r.w[k] = pack2(a[k].x, a[k].y, (T *)nullptr);
    }
    return r;
}

}  // namespace gconv
