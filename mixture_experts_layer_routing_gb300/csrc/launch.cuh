// Kernel launch with programmatic dependent launch: the kernel may be scheduled while its
// predecessor in the stream is finishing. Every kernel launched this way calls griddep_wait()
// (common.cuh) before its first global memory access, which returns once the predecessor grid has
// completed and its writes are visible, so only launch latency and pure prologue overlap; and then
// griddep_launch(), which lets its own successor be scheduled. (After a kernel launched without the
// attribute, or as a kernel's first grid, the wait returns at once.)
#pragma once
#include <cuda_runtime.h>

// Return the error of a launch (or other runtime call) from the enclosing function.
#define MOE_TRY(expr)                          \
  do {                                         \
    const cudaError_t e_ = (expr);             \
    if (e_ != cudaSuccess) return e_;          \
  } while (0)

namespace moe {

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
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
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

}  // namespace moe
