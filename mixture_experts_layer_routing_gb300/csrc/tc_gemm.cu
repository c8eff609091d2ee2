// tcgen05 grouped GEMMs (bf16). Not yet enabled: tc_supported() reports false
// and the bf16 path runs on the CUDA-core kernels.
#include "kernels.h"

namespace moe {
bool tc_supported(const Layer&) { return false; }
cudaError_t tc_init(Layer&) { return cudaErrorNotSupported; }
cudaError_t launch_tc_router_logits(const Layer&, const void*, int, float*, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_tc_gateup(const Layer&, const Bufs&, const void*, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_tc_down(const Layer&, const Bufs&, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_tc_bwd_dh(const Layer&, const Bufs&, const void*, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_tc_bwd_dx(const Layer&, const Bufs&, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_tc_bwd_dw(const Layer&, const Bufs&, const void*, const void*, void*, void*, void*, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace moe
