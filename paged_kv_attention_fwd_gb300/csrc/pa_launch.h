// pa_launch.h -- programmatic dependent launch (griddepcontrol) for the
// kernels that use it.
//
// A kernel launched with programmatic stream serialization may be scheduled
// while the kernel before it in the stream is still running.  It runs its
// shared-memory-only prologue (barrier setup, zero fills) meanwhile and calls
// grid_dependency_wait() before its first access to global memory or its TMEM
// allocation: the wait returns once the previous kernel has completed and its
// memory operations are visible (at once when the launch has no such
// predecessor), so stream order holds for every byte the kernel reads or
// writes.  A kernel that calls allow_dependents_launch() lets such a
// dependent be scheduled once every one of its CTAs has issued the call or
// exited.  Under stream capture the launch becomes a programmatic edge of the
// graph.
#pragma once

#include <utility>
#include <cuda_runtime.h>

namespace pa {

__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void allow_dependents_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... P, typename... A>
cudaError_t launch_overlapped(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              A&&... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}

}  // namespace pa
