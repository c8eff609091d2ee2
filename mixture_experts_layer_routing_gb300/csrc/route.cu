// Routing: router logits (CUDA-core path), top-k selection and gates, expert
// counts, offsets and the stable dispatch permutation, all on the device.
//
// Follows "Cursor открыл код ядра Mixture of Experts ..." (dzen.guru), section
// "Что именно тормозило обучение MoE-моделей?" (each layer routes every token
// to experts) and section "Три решения, которые дали результат" (the CPU is
// out of the loop and sizes no buffer; nothing is dropped; deterministic).
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {

// ---------------------------------------------------------------- logits
// l[t, e] = sum_i x[t, i] Wr[e, i], fp32 accumulation in a fixed order.
// CUDA-core kernel: one warp per (token, 4 experts); used for the fp32
// precision (the bf16 path computes logits on the tensor cores).
template <typename T>
__global__ void __launch_bounds__(256) router_logits_kernel(const T* __restrict__ x, const T* __restrict__ Wr,
                                                            float* __restrict__ logits, int Tn, int d, int E) {
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
    router_logits_kernel<float><<<blocks, 256, 0, s>>>((const float*)x, (const float*)L.Wr, logits, T, L.d, L.E);
  else
    router_logits_kernel<bf16><<<blocks, 256, 0, s>>>((const bf16*)x, (const bf16*)L.Wr, logits, T, L.d, L.E);
  return cudaGetLastError();
}

// ----------------------------------------------------------------- top-k
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits, const float* __restrict__ bias,
                                                   int Tn, int E, int k, int router, int renorm, float scale,
                                                   int* __restrict__ idx, float* __restrict__ gate) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= Tn) return;
  warp_topk_gates(logits + (size_t)t * E, bias, E, k, router, renorm, scale, idx + (size_t)t * k,
                  gate ? gate + (size_t)t * k : nullptr);
}

cudaError_t launch_topk(const Layer& L, const float* logits, int T, int* idx, float* gate, cudaStream_t s) {
  const int blocks = (T * 32 + 255) / 256;
  topk_kernel<<<blocks, 256, 0, s>>>(logits, L.bias, T, L.E, L.k, L.router, L.renorm, L.scale, idx, gate);
  return cudaGetLastError();
}

// ----------------------------------------------- histogram, scan, permute
// Assignments a = t*k + j are cut into chunks of kChunk. (1) each chunk counts
// its experts; (2) one block turns the chunk counts into expert counts, the
// exclusive offsets, per-chunk bases and the M-tile prefix; (3) each chunk
// ranks its assignments stably (warp match + per-warp counts) and writes the
// permutation. Integer-only and order-independent: bit-exact every run.
__global__ void __launch_bounds__(256) hist_kernel(const int* __restrict__ idx, int A, int E,
                                                   int* __restrict__ chunk_hist, int* status) {
  __shared__ int h[kMaxE];
  for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
  __syncthreads();
  const int a0 = blockIdx.x * kChunk;
  for (int a = a0 + threadIdx.x; a < min(A, a0 + kChunk); a += blockDim.x) {
    const int e = idx[a];
    if ((unsigned)e >= (unsigned)E) {
      set_error(status, MOE_ERR_DEVICE_INDEX);
      continue;
    }
    atomicAdd(&h[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_hist[(size_t)blockIdx.x * E + e] = h[e];
}

// One block of 512 threads (E + S <= 512). Segments 0..E-1 are the routed experts, segment E
// (when S = 1) is the shared expert with all T tokens.
__global__ void __launch_bounds__(512) scan_kernel(const int* __restrict__ chunk_hist, int nch, int E, int S, int T,
                                                   int* __restrict__ chunk_base, int* __restrict__ cnt,
                                                   int* __restrict__ off, int* __restrict__ mt_off) {
  __shared__ int c_s[kMaxE + 1];
  __shared__ int warp_tot[16][7];
  __shared__ int tot[4];   // all tiles, candidate dense tiles, other tiles, other non-empty segments
  const int tid = threadIdx.x;
  const int nseg = E + S;
  if (tid < 4) tot[tid] = 0;
  int c = 0;
  if (tid < E) {
    for (int ch = 0; ch < nch; ++ch) c += chunk_hist[(size_t)ch * E + tid];
  } else if (tid == E && S) {
    c = T;
  }
  const int lane = tid & 31, w = tid >> 5;
  const int tiles = (c + kBM - 1) / kBM, pairs = (tiles + 1) / 2;
  // The GEMM schedule interleaves the tiles of "dense" segments (tensor-bound) with the others
  // (HBM-bound) only when that mixes two kinds of work: the candidates (>= kDenseTiles tiles) hold
  // at least a quarter of the tiles and the other non-empty segments average under 1.5 tiles
  // (<= 192 rows per weight byte pair). Otherwise no segment is dense and the order stays
  // segment-major; e.g. uniform routing with 2-3 tiles per expert has both kinds near the ridge.
  const bool cand = tiles >= kDenseTiles;
  __syncthreads();
  if (tiles) {
    atomicAdd(&tot[0], tiles);
    atomicAdd(&tot[cand ? 1 : 2], tiles);
    if (!cand) atomicAdd(&tot[3], 1);
  }
  __syncthreads();
  const bool mix = 4 * tot[1] >= tot[0] && 2 * tot[2] < 3 * tot[3];
  // exclusive scans over the 512 threads of: c, ceil(c / kBM) (tiles), ceil(tiles / 2) (pairs),
  // the tiles of dense segments and of the others, and the same split of the pairs (the GEMMs
  // whose CTAs take two 128-row tiles of a segment at once)
  const int dense = mix && cand ? tiles : 0, sparse = tiles - dense;
  const int dense_p = mix && cand ? pairs : 0, sparse_p = pairs - dense_p;
  constexpr int NQ = 7;
  int v[NQ] = {c, tiles, pairs, dense, sparse, dense_p, sparse_p};
  const int own[NQ] = {c, tiles, pairs, dense, sparse, dense_p, sparse_p};
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const int n = __shfl_up_sync(0xffffffffu, v[q], o);
      if (lane >= o) v[q] += n;
    }
  }
  if (lane == 31) {
#pragma unroll
    for (int q = 0; q < NQ; ++q) warp_tot[w][q] = v[q];
  }
  __syncthreads();
  int ex[NQ];
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    int b = 0;
    for (int u = 0; u < w; ++u) b += warp_tot[u][q];
    ex[q] = b + v[q] - own[q];
  }
  // mt_off, then (kPrefixArrays arrays of nseg + 1 each) the pair prefix, the dense-tile and
  // sparse-tile prefixes, the dense-pair and sparse-pair prefixes
  if (tid < nseg) {
    cnt[tid] = c;
    off[tid] = ex[0];
#pragma unroll
    for (int q = 1; q < NQ; ++q) mt_off[(q - 1) * (nseg + 1) + tid] = ex[q];
    c_s[tid] = ex[0];
  }
  if (tid == nseg - 1) {
    off[nseg] = ex[0] + c;
#pragma unroll
    for (int q = 1; q < NQ; ++q) mt_off[(q - 1) * (nseg + 1) + nseg] = ex[q] + own[q];
  }
  __syncthreads();
  if (tid < E) {
    int run = c_s[tid];
    for (int ch = 0; ch < nch; ++ch) {
      chunk_base[(size_t)ch * E + tid] = run;
      run += chunk_hist[(size_t)ch * E + tid];
    }
  }
}

__global__ void __launch_bounds__(1024) permute_kernel(const int* __restrict__ idx, const float* __restrict__ gate,
                                                       int A, int E, int k, const int* __restrict__ chunk_base,
                                                       int* __restrict__ perm, int* __restrict__ inv,
                                                       int* __restrict__ row_token, float* __restrict__ row_gate) {
  __shared__ int wcnt[32][kMaxE];        // per-warp count of each expert in this chunk
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  for (int i = tid; i < 32 * kMaxE; i += 1024) (&wcnt[0][0])[i] = 0;
  __syncthreads();
  const int a = blockIdx.x * kChunk + tid;
  const bool valid = a < A;
  int e = valid ? idx[a] : -1;
  if (valid && (unsigned)e >= (unsigned)E) e = -1;   // reported by hist_kernel
  const unsigned same = __match_any_sync(0xffffffffu, e);
  const int rank_in_warp = __popc(same & ((1u << lane) - 1u));
  if (e >= 0 && rank_in_warp == 0) wcnt[w][e] = __popc(same);
  __syncthreads();
  if (e >= 0) {
    int before = 0;
    for (int q = 0; q < w; ++q) before += wcnt[q][e];
    const int p = chunk_base[(size_t)blockIdx.x * E + e] + before + rank_in_warp;
    perm[p] = a;
    inv[a] = p;
    row_token[p] = a / k;
    row_gate[p] = gate ? gate[a] : 1.0f;
  }
}

// Shared-expert rows: sorted row A + t is token t with gate 1.
__global__ void shared_rows_kernel(int A, int T, int* __restrict__ row_token, float* __restrict__ row_gate) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t < T) {
    row_token[A + t] = t;
    row_gate[A + t] = 1.0f;
  }
}

cudaError_t launch_scan_permute(const Layer& L, const Bufs& B, cudaStream_t s) {
  hist_kernel<<<B.nch, 256, 0, s>>>(B.idx, B.A, L.E, B.chunk_hist, L.status);
  scan_kernel<<<1, 512, 0, s>>>(B.chunk_hist, B.nch, L.E, L.S, B.T, B.chunk_base, B.cnt, B.off, B.mt_off);
  permute_kernel<<<B.nch, 1024, 0, s>>>(B.idx, B.gate, B.A, L.E, L.k, B.chunk_base, B.perm, B.inv,
                                        B.row_token, B.row_gate);
  if (L.S) shared_rows_kernel<<<(B.T + 255) / 256, 256, 0, s>>>(B.A, B.T, B.row_token, B.row_gate);
  return cudaGetLastError();
}

}  // namespace moe
