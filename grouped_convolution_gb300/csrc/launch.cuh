// launch.cuh -- kernel launches with programmatic dependent launch (PDL).
//
// Every kernel of the library is launched with the programmatic stream
// serialization attribute.  On the device each kernel first allows the next
// kernel in the stream to start launching (pdl_launch_dependents) and then
// waits for the previous kernel's memory to be complete and visible
// (pdl_wait) before its first global-memory access.  The next launch's
// latency and the CTAs' start-up then overlap the tail of the current
// kernel, while a kernel that reads the previous kernel's output still sees
// all of it.  A kernel launched without the attribute, or behind a kernel
// that never signals, simply waits for the previous kernel to finish.
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

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
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
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace gconv
