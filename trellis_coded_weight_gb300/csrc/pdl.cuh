// pdl.cuh -- programmatic dependent launch: a kernel launched with it may be scheduled while the kernel ahead
// of it on the stream is still running, and waits in hardware for that kernel's completion (and its memory
// operations) before it reads or writes global memory.  This hides the gap between back-to-back launches.
#pragma once
#include <cuda_runtime.h>

namespace trellis {

// First statement of a kernel launched with launch_pdl: block until every grid ahead of this one on the stream
// has completed and its writes are visible (a no-op when launched without the attribute), then let the next
// grid be scheduled.  Every CTA of this grid has started once all of them pass this point, so a next grid
// that occupies the free slots cannot keep any CTA of this one from running.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch `kern` on `st` with programmatic stream serialization allowed.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

}  // namespace trellis
