// launch.cuh -- programmatic dependent launch for the short kernels of the
// scale, quantise and forward chains.
//
// A kernel launched with launch_pdl() may be scheduled while the kernel before
// it on the stream is still finishing, which hides its launch latency behind
// that kernel's tail.  Every such kernel calls pdl_wait() before its first
// global-memory access: the wait returns once the preceding kernel has
// completed and its writes are visible, so the stream order of every read and
// write is unchanged.  A kernel may call pdl_trigger() to let its successor be
// scheduled early; that only moves the successor's launch, never its wait.
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace repro {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

} // namespace repro
