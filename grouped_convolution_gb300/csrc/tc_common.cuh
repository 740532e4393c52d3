// tc_common.cuh -- small device helpers shared by the tcgen05 kernels:
// shared-memory matrix and instruction descriptors, bounded mbarrier waits
// (per thread and per converged warp), tensor-core issue through lane 0 of
// a converged warp, TMA issue, tensor-memory loads and fences.  Every wait
// gives up after kTcSpinLimit polls and reports it through the caller's
// failure flag instead of hanging.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace gconv {
namespace tc {

constexpr uint32_t kTcSpinLimit = 1u << 22;

// 64-bit shared-memory matrix descriptor (tcgen05): K-major, no swizzle;
// start address, leading byte offset (between the two K-adjacent 8x16-byte
// core matrices), stride byte offset (between M/N-adjacent ones), in 16-byte
// units; bit 46 holds the descriptor version.
__device__ __forceinline__ uint64_t s_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo & 0x3FFFFu) >> 4) << 16) |
           ((uint64_t)((sbo & 0x3FFFFu) >> 4) << 32) | ((uint64_t)1 << 46);
}

// kind::f16 instruction descriptor: fp32 accumulator, A and B both bf16 or
// both fp16, both K-major, N / 8 and M / 16.
inline uint32_t s_idesc(bool bf16, int M, int N) {
    const uint32_t ab = bf16 ? 1u : 0u;
    return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ bool s_wait(uint32_t bar, uint32_t parity, volatile int *failed) {
    for (uint32_t i = 0; i < kTcSpinLimit; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
        if (*failed) return false;
    }
    *failed = 1;
    return false;
}
// The same wait, bounded but ignoring the failure flag (the clean-up path).
__device__ __forceinline__ void s_wait_final(uint32_t bar, uint32_t parity) {
    for (uint32_t i = 0; i < kTcSpinLimit; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return;
    }
}
// The same wait by a whole warp: every lane polls and the warp leaves the
// loop together, so the code after it stays warp-uniform.
__device__ __forceinline__ bool s_wait_warp(uint32_t bar, uint32_t parity, volatile int *failed) {
    for (uint32_t i = 0; i < kTcSpinLimit; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (__all_sync(0xffffffffu, done != 0)) return true;
        if (__any_sync(0xffffffffu, *failed != 0)) return false;
    }
    *failed = 1;
    return false;
}
__device__ __forceinline__ void s_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void s_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void s_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
// Issue forms for a converged warp: lane 0 issues, the other lanes pass
// over the predicated instruction, so the warp never diverges around the
// issue and its operands stay warp-uniform.
__device__ __forceinline__ void s_mma_lane0(uint32_t tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, int accumulate, uint32_t lane) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\tsetp.eq.u32 e, %5, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(lane));
}
__device__ __forceinline__ void s_commit_lane0(uint32_t bar, uint32_t lane) {
    asm volatile(
        "{\n\t.reg .pred e;\n\tsetp.eq.u32 e, %1, 0;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}\n" ::"r"(bar),
        "r"(lane)
        : "memory");
}
__device__ __forceinline__ void s_expect_tx_lane0(uint32_t bar, uint32_t bytes, uint32_t lane) {
    asm volatile(
        "{\n\t.reg .pred e;\n\tsetp.eq.u32 e, %2, 0;\n\t"
        "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}\n" ::"r"(bar),
        "r"(bytes), "r"(lane)
        : "memory");
}
__device__ __forceinline__ void s_tma_lane0(uint32_t dst, const CUtensorMap *map, uint32_t bar, int c0,
                                            int c1, int c2, int c3, uint32_t lane) {
    asm volatile(
        "{\n\t.reg .pred e;\n\tsetp.eq.u32 e, %7, 0;\n\t"
        "@e cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%3, %4, %5, %6}], [%2];\n\t}\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(lane)
        : "memory");
}
template <int NC>
__device__ __forceinline__ void s_ld(uint32_t taddr, float (&v)[NC]);
template <>
__device__ __forceinline__ void s_ld<8>(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
template <>
__device__ __forceinline__ void s_ld<16>(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
        "[%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
template <>
__device__ __forceinline__ void s_ld<4>(uint32_t taddr, float (&v)[4]) {
    uint32_t r[4];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void s_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}
}  // namespace tc
}  // namespace gconv
