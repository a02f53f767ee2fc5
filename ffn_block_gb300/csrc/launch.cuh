// Kernel launches with programmatic dependent launch.
//
// Every kernel of the library is launched with programmatic stream
// serialization allowed, and starts with pdl_enter(): it lets the next kernel
// of the stream begin launching, then waits until the kernels before it have
// completed and their writes are visible.  So a kernel's CTAs are dispatched
// while the previous kernel's last wave is still running, and start work the
// moment it completes, instead of after the launch gap.  Nothing a kernel
// reads or writes in global memory is touched before its pdl_enter() (or
// pdl_wait()), so the order of the stream's kernels is unchanged.
#pragma once

#include <cuda_runtime.h>

namespace rmx {

// Lets the next grid of the stream launch (its CTAs still wait in
// pdl_wait() for this grid to complete).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// Waits until the previous grids of the stream have completed and their
// memory operations are visible; returns at once when there are none.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_enter() {
  pdl_trigger();
  pdl_wait();
}

// Launches k<<<grid, block, smem, st>>>(args...) with programmatic stream
// serialization allowed, and clusters of cluster_x CTAs along x when
// cluster_x > 1.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, unsigned cluster_x,
                     Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, k, static_cast<KArgs>(args)...);
}

}  // namespace rmx
