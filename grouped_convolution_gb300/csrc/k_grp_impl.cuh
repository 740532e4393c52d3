// k_grp_impl.cuh -- launch of grp_kernel for one dtype (included by the
// per-dtype translation units).
#pragma once

#include "k_grp.cuh"

namespace gconv {

template <typename T, int CIP, int MB, int SW>
cudaError_t grp_launch_t(const Params &p, const Ptrs &q, cudaStream_t s, const GrpGeom &g) {
    const size_t smem = grp_smem_bytes(p, g, CIP);
    cudaError_t e = cudaFuncSetAttribute(grp_kernel<T, CIP, MB, SW>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_kernel(grp_kernel<T, CIP, MB, SW>, dim3((unsigned)g.tiles), dim3(kGrpThreads), smem, s,
                   static_cast<const T *>(q.x), static_cast<const T *>(q.w),
                   static_cast<const T *>(q.b), static_cast<T *>(q.y), p, g);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename T, int CIP, int MB>
cudaError_t grp_launch_sw(const Params &p, const Ptrs &q, cudaStream_t s, const GrpGeom &g) {
    return p.sw == 1 ? grp_launch_t<T, CIP, MB, 1>(p, q, s, g)
                     : grp_launch_t<T, CIP, MB, 2>(p, q, s, g);
}

template <typename T>
cudaError_t grp_launch_dtype(const Params &p, const Ptrs &q, cudaStream_t s) {
    const int es = (int)sizeof(T);
    GrpGeom g;
    int cip, mb;
    if (!grp_geometry(p, es, g, cip, mb)) return cudaErrorNotSupported;
    // One cp.async per pixel: channels-last, all CIP slots real, 8/16 bytes,
    // every pixel run aligned to its size.
    const int px_bytes = p.Cin_g * es;
    const uintptr_t xa = reinterpret_cast<uintptr_t>(q.x);
    g.vec_load = p.layout == GCONV_LAYOUT_NHWC && p.Cin_g == cip &&
                 (px_bytes == 8 || px_bytes == 16) && xa % px_bytes == 0 &&
                 (p.xs[0] * es) % px_bytes == 0 && (p.xs[2] * es) % px_bytes == 0 &&
                 (p.xs[3] * es) % px_bytes == 0;
    // MB contiguous output channels per vector store.
    const int vb = mb * es > 16 ? 16 : mb * es;
    const uintptr_t ya = reinterpret_cast<uintptr_t>(q.y);
    g.vec_store = p.ys[1] == 1 && ya % vb == 0 && (p.ys[0] * es) % vb == 0 &&
                  (p.ys[2] * es) % vb == 0 && (p.ys[3] * es) % vb == 0 &&
                  (p.Cout_g * es) % vb == 0;
    if (cip == 4) {
        if (mb == 2) return grp_launch_sw<T, 4, 2>(p, q, s, g);
        if (mb == 4) return grp_launch_sw<T, 4, 4>(p, q, s, g);
        return grp_launch_sw<T, 4, 8>(p, q, s, g);
    }
    if (mb == 2) return grp_launch_sw<T, 8, 2>(p, q, s, g);
    if (mb == 4) return grp_launch_sw<T, 8, 4>(p, q, s, g);
    return grp_launch_sw<T, 8, 8>(p, q, s, g);
}

}  // namespace gconv
