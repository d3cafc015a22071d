// launch.cuh -- kernel launches with programmatic dependent launch.
//
// Every kernel of the library is launched with the programmatic stream
// serialization attribute: the GPU may start scheduling it while the kernel
// before it on the stream is still finishing (each kernel signals this with
// griddepcontrol.launch_dependents as soon as it starts).  The launched
// kernel then runs its set-up (barrier initialisation, tensor-memory
// allocation, descriptor prefetch) and executes griddepcontrol.wait, which
// returns once the previous kernel has completed and its memory is visible,
// before it touches global memory.  Back-to-back calls thus hide the launch
// gap and the set-up of the next kernel.  DGEMM_PDL=0 launches plainly.
#pragma once

#include <cstdlib>
#include <utility>
#include <cuda_runtime.h>

namespace dg {

inline bool pdl_enabled() {
  static const bool on = [] {
    const char *e = std::getenv("DGEMM_PDL");
    return !(e && e[0] == '0');
  }();
  return on;
}

// Launch `kern` with grid x block threads, `smem` bytes of dynamic shared
// memory, on `stream`, in clusters of `cluster` CTAs along x (1 = none).
template <class... KArgs, class... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, unsigned cluster, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (pdl_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Device side: let the next kernel on the stream be scheduled, and wait
// until the previous one has completed (no-ops without the attribute).
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

}  // namespace dg
