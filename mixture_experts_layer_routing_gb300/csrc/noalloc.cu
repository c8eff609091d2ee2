// moe_route_noalloc: routing whose scratch lives in a fixed array inside the
// library, for callers that cannot allocate device memory.
//
// Who needs it: a plugin running inside a host program that owns and budgets
// all device memory and hands its plugins no allocator; a serving loop that
// bans cudaMalloc/cudaFree once it has started, because those calls can block
// and synchronise the whole device in the middle of a latency-bound step;
// small tools that just want routing without sizing and keeping a workspace.
// These callers still pass their input and output buffers; only the scratch
// (per-chunk expert histograms and bases, internal offsets, the row maps of
// the permutation) moves into the array below.
//
// The array is file-scope device memory: every GPU that loads the library
// holds it until the process exits. Host code cannot use its name as a device
// address, so its address is looked up once per device with
// cudaGetSymbolAddress (on that device's first call) and passed to the kernels.
#include <mutex>

#include "common.cuh"
#include "handle.h"
#include "kernels.h"

using namespace moe;

namespace {

constexpr size_t kScratchBytes = size_t(4) << 20;   // 4 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_route_scratch[kScratchBytes];
// split-K partials of the router GEMM (the same splits as every other routing call, so the logits
// are summed in the same order)
static __device__ __align__(256) float g_router_part[kRouterPartBytes / sizeof(float)];

std::mutex g_mu;
void* g_scratch[kMaxDevices] = {};
void* g_part[kMaxDevices] = {};

inline size_t al(size_t v) { return (v + 255) & ~size_t(255); }

// Scratch bytes one routing call of T tokens needs.
size_t scratch_bytes(const Layer& L, int T) {
  const size_t A = (size_t)T * L.k, R = A + (size_t)L.S * T, nseg = L.E + L.S;
  const size_t nch = (A + kChunk - 1) / kChunk;
  return 2 * al(4 * nch * L.E) + 2 * al(4 * (nseg + 1)) + al(4 * kPrefixArrays * (nseg + 1)) + al(4 * R) +
         al(4 * R);
}

// Device addresses of the arrays on device `dev` (the current device): out[0] the routing scratch,
// out[1] the router partials. Looked up on the first call for that device and remembered for the
// life of the process: a cudaDeviceReset (or any teardown of the device's primary context) makes
// the remembered addresses stale, so a process that resets a device must not call this entry
// point on that device afterwards.
cudaError_t scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!g_scratch[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess) return e;
    void* q = nullptr;
    e = cudaGetSymbolAddress(&q, g_router_part);
    if (e != cudaSuccess) return e;
    g_scratch[dev] = p;
    g_part[dev] = q;
  }
  out[0] = g_scratch[dev];
  out[1] = g_part[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" moe_status moe_route_noalloc(moe_handle h, const void* x, int T, float* logits, int32_t* idx,
                                        float* gate, int32_t* cnt, int32_t* off, int32_t* perm, int32_t* inv,
                                        void* stream) {
  if (!h || !x || !logits || !idx || !gate || !cnt || !off || !perm || !inv) return MOE_ERR_INVALID_ARG;
  if (T < 0 || T > h->cfg.T_max) return MOE_ERR_INVALID_ARG;
  if (!h->L.has_weights) return MOE_ERR_NO_WEIGHTS;
  const Layer& L = h->L;
  if (scratch_bytes(L, T) > kScratchBytes) return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev != h->device) return MOE_ERR_INVALID_ARG;
  void* addr[2] = {};
  if (scratch_address(dev, addr) != cudaSuccess) return MOE_ERR_CUDA;
  void* base = addr[0];

  Bufs B = {};
  B.T = T;
  B.A = T * L.k;
  B.R = B.A + L.S * T;
  B.nch = (B.A + kChunk - 1) / kChunk;
  const size_t nseg = L.E + L.S;
  char* p = (char*)base;
  B.chunk_hist = (int*)p; p += al(4 * (size_t)B.nch * L.E);
  B.chunk_base = (int*)p; p += al(4 * (size_t)B.nch * L.E);
  B.cnt = (int*)p; p += al(4 * (nseg + 1));
  B.off = (int*)p; p += al(4 * (nseg + 1));
  B.mt_off = (int*)p; p += al(4 * kPrefixArrays * (nseg + 1));   // mt_off, then the other tile prefixes
  B.row_token = (int*)p; p += al(4 * (size_t)B.R);
  B.row_gate = (float*)p;
  B.logits = logits;
  B.idx = idx;
  B.gate = gate;
  B.perm = perm;
  B.inv = inv;

  cudaStream_t s = (cudaStream_t)stream;
  // Every scratch entry the kernels read is written earlier in the same call,
  // so nothing needs clearing between calls. The steps are moe_route's own
  // (same router path for every precision, same split-K order, same launch
  // counting and profiling records).
  const moe_status st = route_steps(h, B, x, (float*)addr[1], kRouterPartBytes, s);
  if (st != MOE_OK) return st;
  cudaError_t e = cudaMemcpyAsync(cnt, B.cnt, 4 * (size_t)L.E, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(off, B.off, 4 * (size_t)(L.E + 1), cudaMemcpyDeviceToDevice, s);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
