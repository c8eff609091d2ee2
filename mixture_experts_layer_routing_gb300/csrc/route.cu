// Routing: router logits (CUDA-core path), top-k selection and gates, expert
// counts, offsets and the stable dispatch permutation, all on the device.
//
// Follows "Cursor открыл код ядра Mixture of Experts ..." (dzen.guru), section
// "Что именно тормозило обучение MoE-моделей?" (each layer routes every token
// to experts) and section "Три решения, которые дали результат" (the CPU is
// out of the loop and sizes no buffer; nothing is dropped; deterministic).
#include "common.cuh"
#include "kernels.h"
#include "route_phases.cuh"
#include "topk.cuh"
#include "launch.cuh"

namespace moe {

// ---------------------------------------------------------------- logits
// l[t, e] = sum_i x[t, i] Wr[e, i], fp32 accumulation in a fixed order.
// CUDA-core kernel: one warp per (token, 4 experts); used for the fp32
// precision (the bf16 path computes logits on the tensor cores).
template <typename T>
__global__ void __launch_bounds__(256) router_logits_kernel(const T* __restrict__ x, const T* __restrict__ Wr,
                                                            float* __restrict__ logits, int Tn, int d, int E) {
  griddep_wait();    // after the predecessor grid (launch.cuh)
  griddep_launch();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int e_groups = (E + 3) / 4;
  const int t = warp / e_groups;
  const int e0 = (warp % e_groups) * 4;
  if (t >= Tn) return;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const T* xr = x + (size_t)t * d;
  for (int i = lane; i < d; i += 32) {
    const float xv = to_f(xr[i]);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (e0 + q < E) acc[q] = fmaf(xv, to_f(Wr[(size_t)(e0 + q) * d + i]), acc[q]);
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float s = warp_sum(acc[q]);
    if (lane == 0 && e0 + q < E) logits[(size_t)t * E + e0 + q] = s;
  }
}

cudaError_t launch_router_logits(const Layer& L, const void* x, int T, float* logits, cudaStream_t s) {
  const long warps = (long)T * ((L.E + 3) / 4);
  const int blocks = (int)((warps * 32 + 255) / 256);
  if (L.prec == MOE_FP32)
    MOE_TRY(launch_pdl(router_logits_kernel<float>, dim3(blocks), dim3(256), 0, s, (const float*)x,
        (const float*)L.Wr, logits, T, L.d, L.E));
  else
    MOE_TRY(launch_pdl(router_logits_kernel<bf16>, dim3(blocks), dim3(256), 0, s, (const bf16*)x, (const bf16*)L.Wr,
        logits, T, L.d, L.E));
  return cudaGetLastError();
}

// ----------------------------------------------------------------- top-k
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits, const float* __restrict__ bias,
                                                   int Tn, int E, int k, int router, int renorm, float scale,
                                                   int* __restrict__ idx, float* __restrict__ gate) {
  griddep_wait();    // after the predecessor grid (launch.cuh)
  griddep_launch();
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= Tn) return;
  warp_topk_gates(logits + (size_t)t * E, bias, E, k, router, renorm, scale, idx + (size_t)t * k,
                  gate ? gate + (size_t)t * k : nullptr);
}

cudaError_t launch_topk(const Layer& L, const float* logits, int T, int* idx, float* gate, cudaStream_t s) {
  const int blocks = (T * 32 + 255) / 256;
  MOE_TRY(launch_pdl(topk_kernel, dim3(blocks), dim3(256), 0, s, logits, L.bias, T, L.E, L.k, L.router, L.renorm,
      L.scale, idx, gate));
  return cudaGetLastError();
}

// ----------------------------------------------- histogram, scan, permute
// (block-level bodies in route_phases.cuh, shared with the whole-forward persistent kernel)
__global__ void __launch_bounds__(256) hist_kernel(const int* __restrict__ idx, int A, int E,
                                                   int* __restrict__ chunk_hist, int* status) {
  griddep_wait();    // after the predecessor grid (launch.cuh)
  griddep_launch();
  __shared__ int h[kHistSmem];
  hist_chunk(idx, A, E, blockIdx.x, chunk_hist, status, h);
}

// One block of 512 threads (E + S <= 512).
__global__ void __launch_bounds__(512) scan_kernel(const int* __restrict__ chunk_hist, int nch, int E, int S, int T,
                                                   int* __restrict__ chunk_base, int* __restrict__ cnt,
                                                   int* __restrict__ off, int* __restrict__ mt_off) {
  griddep_wait();    // after the predecessor grid (launch.cuh)
  griddep_launch();
  __shared__ int sm[kScanSmem];
  scan_segments(chunk_hist, nch, E, S, T, chunk_base, cnt, off, mt_off, sm);
}

// One block of kChunk threads per chunk (one pass).
__global__ void __launch_bounds__(kChunk) permute_kernel(const int* __restrict__ idx, const float* __restrict__ gate,
                                                         int A, int E, int k, const int* __restrict__ chunk_base,
                                                         int* __restrict__ perm, int* __restrict__ inv,
                                                         int* __restrict__ row_token, float* __restrict__ row_gate) {
  griddep_wait();    // after the predecessor grid (launch.cuh)
  griddep_launch();
  __shared__ int sm[permute_smem(kChunk / 32)];
  permute_chunk(idx, gate, A, E, k, blockIdx.x, chunk_base, perm, inv, row_token, row_gate, sm);
}

// Shared-expert rows: sorted row A + t is token t with gate 1.
__global__ void shared_rows_kernel(int A, int T, int* __restrict__ row_token, float* __restrict__ row_gate) {
  griddep_wait();    // after the predecessor grid (launch.cuh)
  griddep_launch();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t < T) {
    row_token[A + t] = t;
    row_gate[A + t] = 1.0f;
  }
}

cudaError_t launch_scan_permute(const Layer& L, const Bufs& B, cudaStream_t s) {
  MOE_TRY(launch_pdl(hist_kernel, dim3(B.nch), dim3(256), 0, s, B.idx, B.A, L.E, B.chunk_hist, L.status));
  MOE_TRY(launch_pdl(scan_kernel, dim3(1), dim3(512), 0, s, B.chunk_hist, B.nch, L.E, L.S, B.T, B.chunk_base, B.cnt,
      B.off, B.mt_off));
  MOE_TRY(launch_pdl(permute_kernel, dim3(B.nch), dim3(kChunk), 0, s, B.idx, B.gate, B.A, L.E, L.k, B.chunk_base,
      B.perm, B.inv, B.row_token, B.row_gate));
  if (L.S)
    MOE_TRY(launch_pdl(shared_rows_kernel, dim3((B.T + 255) / 256), dim3(256), 0, s, B.A, B.T, B.row_token,
        B.row_gate));
  return cudaGetLastError();
}

}  // namespace moe
