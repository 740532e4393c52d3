// launch.cuh -- kernel launches, optionally with programmatic dependent
// launch (PDL).
//
// On the device each kernel first allows the next kernel in the stream to
// start launching (pdl_launch_dependents) and then waits for the previous
// kernel's memory to be complete and visible (pdl_wait) before its first
// global-memory access.  Both are no-ops unless the kernel was launched with
// the programmatic stream serialization attribute, which the library sets
// only when the environment variable GCONV_PDL is 1 (read once per process).
// Measured on the six-convolution benchmark step (six different kernels back
// to back), the attribute made the step slower, 247 us against 230 us without
// it.  The next kernel's CTAs launch early and wait at griddepcontrol.wait
// while the previous kernel's last CTAs run.  A loop of one kernel gains 2-6 %
// from it instead.
#pragma once

#include <cuda_runtime.h>
#include <utility>

namespace gconv {

__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

bool pdl_enabled();   // GCONV_PDL=1 in the environment (host.cpp)

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace gconv
