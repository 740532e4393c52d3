// tma.cuh -- tensor-memory-accelerator (TMA) row loads with mbarrier
// completion, for sm_100+ kernels.
//
// Host side: a tiled tensor map is encoded through the driver entry point
// cuTensorMapEncodeTiled (resolved once through the runtime, so the library
// does not link the driver library).  Out-of-bounds elements of a box are
// filled with zeros, which is how the stencils get their padding.
//
// Device side: one thread arms an mbarrier with the expected byte count and
// issues the bulk tensor copy; consumers wait on the barrier's phase.  Every
// wait is bounded: after kTmaSpinLimit polls it gives up and reports failure
// to the caller instead of hanging.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <type_traits>

namespace gconv {

constexpr uint32_t kTmaSpinLimit = 1u << 22;

// Encode a rank-4 tiled map over a tensor whose innermost dim is dims[0].
// strides_bytes[i] is the byte stride of dims[i + 1].  Returns false when
// the driver entry point is missing or the encode is rejected.
bool tma_encode_4d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base,
                   const uint64_t dims[4], const uint64_t strides_bytes[3],
                   const uint32_t box[4]);

// The same with a traversal stride per dim: the box spans box[i] elements
// of dim i and loads every element_strides[i]-th of them (box[i] /
// element_strides[i] per dim, packed in shared memory).
bool tma_encode_4d_strided(CUtensorMap *map, CUtensorMapDataType dtype, const void *base,
                           const uint64_t dims[4], const uint64_t strides_bytes[3],
                           const uint32_t box[4], const uint32_t element_strides[4]);

// Tensor-map element type of T (float, __half or __nv_bfloat16).
template <typename T> constexpr CUtensorMapDataType tma_dtype() {
    return sizeof(T) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                          : (std::is_same<T, __half>::value ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                            : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count));
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

// Poll the barrier until the phase with the given parity has completed.
// Returns false if it did not complete within kTmaSpinLimit polls, or, when
// `abort` is given, as soon as *abort is set after the first 64 polls (the
// flag is read only on that slow path).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          const volatile int *abort = nullptr) {
    for (uint32_t i = 0; i < kTmaSpinLimit; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
        if (abort && i >= 64 && *abort) return false;
    }
    return false;
}

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Copy the box at coordinates (c0, c1, c2, c3) into shared memory at dst and
// signal completion (bytes) on bar.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%3, %4, %5, %6}], [%2];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

}  // namespace gconv
