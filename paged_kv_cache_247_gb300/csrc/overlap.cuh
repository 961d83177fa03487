// Programmatic dependent launch for the decode and cache-maintenance
// kernels.  sm_90 and later.
#pragma once

#include <cuda_runtime.h>

namespace pkv {

// Programmatic dependent launch.  A kernel launched by launch_overlapped()
// may be resident while the previous kernel on its stream still runs.
// grid_dep_wait() returns once that kernel has finished and its writes are
// visible (at once when the launch had no such overlap).  Every overlapped
// kernel calls it first, in every thread and before any early return, so a
// kernel's completion still implies its predecessor's along a chain.
// grid_dep_launch_dependents() lets the next overlapped kernel's CTAs be
// placed on SMs this grid leaves idle; they wait in their own grid_dep_wait().
__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_dep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch with programmatic stream serialization (see grid_dep_wait).
template <typename... Params, typename... Args>
cudaError_t launch_overlapped(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
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
  const cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, args...);
  const cudaError_t last = cudaGetLastError();  // clears the error, as after <<<>>>
  return err != cudaSuccess ? err : last;
}

}  // namespace pkv
