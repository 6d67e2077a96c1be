// Programmatic dependent launch for the selection's chain of kernels on one stream.
//
// A kernel launched with launch_pdl may start while the kernel before it on the stream is
// still draining: its CTAs are scheduled once every CTA of that kernel has signalled
// pdl_trigger() (or exited), and pdl_wait() then blocks until that kernel has completed and
// its memory writes are visible.  Each kernel of the chain therefore calls pdl_wait() before
// it reads or writes anything, and pdl_trigger() at its start so that the next one's launch
// overlaps its run.  Both instructions are no-ops for a kernel launched without the attribute.
// The trigger only lets the next grid launch: since it fires once all CTAs of this grid are
// resident, the next grid's waiting CTAs can never keep one of this grid's CTAs off an SM.
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace pisa {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
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
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace pisa
