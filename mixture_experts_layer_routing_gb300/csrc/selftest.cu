// Device-side failure path self-test: a pipeline wait that can never be satisfied.
//
// One block initialises an mbarrier that nothing ever arrives at and waits on
// it with the bounded wait every tcgen05 pipeline of the library uses, here
// with a caller-chosen short limit. Past the limit the wait records
// MOE_ERR_TIMEOUT in the handle's status word and the kernel returns, so the
// context stays usable. Nothing faults, traps or hangs.
#include "common.cuh"
#include "handle.h"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {
__global__ void selftest_wait_kernel(uint64_t limit_ns, int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, status, limit_ns);
}
}  // namespace
}  // namespace moe

extern "C" moe_status moe_selftest_timeout(moe_handle h, int limit_ms, void* stream) {
  if (!h || limit_ms < 1 || limit_ms > 10000) return MOE_ERR_INVALID_ARG;
  moe::selftest_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((uint64_t)limit_ms * 1000000ull, h->L.status);
  h->launches += 1;
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
