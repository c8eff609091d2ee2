// CUDA-core grouped GEMMs of the expert FFN, forward and backward.
//
// These kernels serve the fp32 precision (small layers, launch-bound) and any
// shape the tensor-core path does not take. Every sum runs in a fixed order
// (fp32 accumulation along K in ascending order), so results are bit-identical
// between runs. Tokens are pulled by index from x (the dispatch never
// materialises a permuted copy of x), following the pull dispatch of
// "Cursor открыл код ядра Mixture of Experts ..." (dzen.guru), section
// "Три решения, которые дали результат".
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int TM = 64, TN = 64, TK = 16;

// 64x64 output tile, 256 threads, each 4x4. a_at(m, k) and b_at(k, n) return
// the operand (0 outside the problem).
template <class AF, class BF>
__device__ __forceinline__ void tile_mma(const AF& a_at, const BF& b_at, int K, float (&acc)[4][4],
                                         float (*sA)[TM], float (*sB)[TN]) {
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  for (int k0 = 0; k0 < K; k0 += TK) {
    for (int i = tid; i < TM * TK; i += 256) {
      const int m = i / TK, kk = i % TK;
      sA[kk][m] = (k0 + kk < K) ? a_at(m, k0 + kk) : 0.f;
    }
    for (int i = tid; i < TN * TK; i += 256) {
      const int n = i / TK, kk = i % TK;
      sB[kk][n] = (k0 + kk < K) ? b_at(k0 + kk, n) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = sA[kk][ty * 4 + i];
        b[i] = sB[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
}

// Maps a 64-row tile index to (segment, first row, segment end) through the
// 128-row M-tile prefix mt_off. Returns false past the last tile.
__device__ __forceinline__ bool map_rows64(const int* mt_off, const int* off, int nseg, int tile64, int& e,
                                           int& row0, int& row_end) {
  const int t128 = tile64 >> 1;
  if (t128 >= mt_off[nseg]) return false;
  int lo = 0, hi = nseg;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (mt_off[mid] <= t128) lo = mid; else hi = mid;
  }
  e = lo;
  row0 = off[e] + (t128 - mt_off[e]) * kBM + (tile64 & 1) * TM;
  row_end = off[e + 1];
  return row0 < row_end;
}

// packed W13 row of gate feature i (is_up = 0) or up feature i (is_up = 1)
__device__ __forceinline__ int w13_row(int i, int G, int is_up) { return (i / G) * 2 * G + (i % G) + is_up * G; }

template <typename T>
__global__ void __launch_bounds__(256) gateup_kernel(const T* __restrict__ x, const T* __restrict__ W13,
                                                     const int* __restrict__ off, const int* __restrict__ mt_off,
                                                     const int* __restrict__ row_token, int nseg, int d, int f, int G,
                                                     T* __restrict__ h, T* __restrict__ uv) {
  __shared__ float sA[TK][TM], sB[TK][TN];
  __shared__ float sC[TM][TN + 1];
  int e, row0, row_end;
  if (!map_rows64(mt_off, off, nseg, blockIdx.x, e, row0, row_end)) return;
  const int i0 = blockIdx.y * 32;
  const T* We = W13 + (size_t)e * 2 * f * d;
  auto a_at = [&](int m, int k) -> float {
    const int r = row0 + m;
    return r < row_end ? to_f(x[(size_t)row_token[r] * d + k]) : 0.f;
  };
  auto b_at = [&](int k, int n) -> float {
    return to_f(We[(size_t)w13_row(i0 + (n & 31), G, n >> 5) * d + k]);
  };
  float acc[4][4] = {};
  tile_mma(a_at, b_at, d, acc, sA, sB);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) sC[ty * 4 + i][tx * 4 + j] = acc[i][j];
  __syncthreads();
  for (int q = threadIdx.x; q < TM * 32; q += 256) {
    const int m = q >> 5, c = q & 31, r = row0 + m;
    if (r >= row_end) continue;
    const float u = sC[m][c], v = sC[m][32 + c];
    h[(size_t)r * f + i0 + c] = from_f<T>(silu_f(u) * v);
    if (uv) {
      uv[(size_t)r * 2 * f + w13_row(i0 + c, G, 0)] = from_f<T>(u);
      uv[(size_t)r * 2 * f + w13_row(i0 + c, G, 1)] = from_f<T>(v);
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256) down_kernel(const T* __restrict__ h, const T* __restrict__ Wd,
                                                   const int* __restrict__ off, const int* __restrict__ mt_off,
                                                   const float* __restrict__ row_gate, int nseg, int d, int f,
                                                   T* __restrict__ o) {
  __shared__ float sA[TK][TM], sB[TK][TN];
  int e, row0, row_end;
  if (!map_rows64(mt_off, off, nseg, blockIdx.x, e, row0, row_end)) return;
  const int c0 = blockIdx.y * TN;
  const T* We = Wd + (size_t)e * d * f;
  auto a_at = [&](int m, int k) -> float { return row0 + m < row_end ? to_f(h[(size_t)(row0 + m) * f + k]) : 0.f; };
  auto b_at = [&](int k, int n) -> float { return c0 + n < d ? to_f(We[(size_t)(c0 + n) * f + k]) : 0.f; };
  float acc[4][4] = {};
  tile_mma(a_at, b_at, f, acc, sA, sB);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = row0 + ty * 4 + i;
    if (r >= row_end) continue;
    const float g = row_gate[r];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = c0 + tx * 4 + j;
      if (c < d) o[(size_t)r * d + c] = from_f<T>(g * acc[i][j]);
    }
  }
}

// r = dy_t Wd[e] (K = d), then the SwiGLU backward and the gate gradient partial.
template <typename T>
__global__ void __launch_bounds__(256) bwd_dh_kernel(const T* __restrict__ dy, const T* __restrict__ Wd,
                                                     const T* __restrict__ uv, const int* __restrict__ off,
                                                     const int* __restrict__ mt_off, const int* __restrict__ row_token,
                                                     const float* __restrict__ row_gate, int nseg, int A, int d, int f,
                                                     int G, T* __restrict__ dudv, T* __restrict__ hg,
                                                     float* __restrict__ dg_part) {
  __shared__ float sA[TK][TM], sB[TK][TN];
  __shared__ float sC[TM][TN + 1];
  int e, row0, row_end;
  if (!map_rows64(mt_off, off, nseg, blockIdx.x, e, row0, row_end)) return;
  const int i0 = blockIdx.y * TN;
  const T* We = Wd + (size_t)e * d * f;
  auto a_at = [&](int m, int k) -> float {
    const int r = row0 + m;
    return r < row_end ? to_f(dy[(size_t)row_token[r] * d + k]) : 0.f;
  };
  auto b_at = [&](int k, int n) -> float { return to_f(We[(size_t)k * f + i0 + n]); };
  float acc[4][4] = {};
  tile_mma(a_at, b_at, d, acc, sA, sB);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) sC[ty * 4 + i][tx * 4 + j] = acc[i][j];
  __syncthreads();
  // each thread: one row m (64 rows x 4 threads), 16 features; fixed-order partial sums
  const int m = threadIdx.x >> 2, part = threadIdx.x & 3;
  const int r = row0 + m;
  float dg = 0.f;
  if (r < row_end) {
    const float g = row_gate[r];
    for (int c = part * 16; c < part * 16 + 16; ++c) {
      const int i = i0 + c;
      const float u = to_f(uv[(size_t)r * 2 * f + w13_row(i, G, 0)]);
      const float v = to_f(uv[(size_t)r * 2 * f + w13_row(i, G, 1)]);
      const float rr = sC[m][c];
      const float su = sigmoid_f(u);
      const float sl = u * su;
      const float hv = sl * v;
      dg = fmaf(rr, hv, dg);
      const float dh = g * rr;
      dudv[(size_t)r * 2 * f + w13_row(i, G, 0)] = from_f<T>(dh * v * su * (1.f + u * (1.f - su)));
      dudv[(size_t)r * 2 * f + w13_row(i, G, 1)] = from_f<T>(dh * sl);
      hg[(size_t)r * f + i] = from_f<T>(g * hv);
    }
  }
  dg += __shfl_down_sync(0xffffffffu, dg, 1, 4);
  dg += __shfl_down_sync(0xffffffffu, dg, 2, 4);
  if (part == 0 && r < row_end && r < A) dg_part[(size_t)r * (f / TN) + blockIdx.y] = dg;
}

// dx_rows[p] = dudv[p] W13[e] (K = 2f)
template <typename T>
__global__ void __launch_bounds__(256) bwd_dx_kernel(const T* __restrict__ dudv, const T* __restrict__ W13,
                                                     const int* __restrict__ off, const int* __restrict__ mt_off,
                                                     int nseg, int d, int f, T* __restrict__ dx_rows) {
  __shared__ float sA[TK][TM], sB[TK][TN];
  int e, row0, row_end;
  if (!map_rows64(mt_off, off, nseg, blockIdx.x, e, row0, row_end)) return;
  const int c0 = blockIdx.y * TN;
  const T* We = W13 + (size_t)e * 2 * f * d;
  auto a_at = [&](int m, int k) -> float {
    return row0 + m < row_end ? to_f(dudv[(size_t)(row0 + m) * 2 * f + k]) : 0.f;
  };
  auto b_at = [&](int k, int n) -> float { return c0 + n < d ? to_f(We[(size_t)k * d + c0 + n]) : 0.f; };
  float acc[4][4] = {};
  tile_mma(a_at, b_at, 2 * f, acc, sA, sB);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = row0 + ty * 4 + i;
    if (r >= row_end) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = c0 + tx * 4 + j;
      if (c < d) dx_rows[(size_t)r * d + c] = from_f<T>(acc[i][j]);
    }
  }
}

// dW13[e] = dudv_seg^T x_seg and dWd[e] = dy_seg^T hg_seg, K = the segment's rows in sorted order.
template <typename T>
__global__ void __launch_bounds__(256) bwd_dw13_kernel(const T* __restrict__ dudv, const T* __restrict__ x,
                                                       const int* __restrict__ off, const int* __restrict__ row_token,
                                                       int d, int f, int G, int accumulate, T* __restrict__ dWg,
                                                       T* __restrict__ dWu) {
  __shared__ float sA[TK][TM], sB[TK][TN];
  const int e = blockIdx.z, r0 = blockIdx.y * TM, c0 = blockIdx.x * TN;
  const int p0 = off[e], K = off[e + 1] - off[e];
  auto a_at = [&](int m, int k) -> float { return to_f(dudv[(size_t)(p0 + k) * 2 * f + r0 + m]); };
  auto b_at = [&](int k, int n) -> float {
    return c0 + n < d ? to_f(x[(size_t)row_token[p0 + k] * d + c0 + n]) : 0.f;
  };
  float acc[4][4] = {};
  tile_mma(a_at, b_at, K, acc, sA, sB);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int pr = r0 + ty * 4 + i;                 // packed row
    const int blk = pr / (2 * G), w = pr % (2 * G);
    const int feat = blk * G + (w % G);
    T* dst = (w < G ? dWg : dWu) + ((size_t)e * f + feat) * d;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = c0 + tx * 4 + j;
      if (c < d) dst[c] = from_f<T>(accumulate ? acc[i][j] + to_f(dst[c]) : acc[i][j]);
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256) bwd_dwd_kernel(const T* __restrict__ dy, const T* __restrict__ hg,
                                                      const int* __restrict__ off, const int* __restrict__ row_token,
                                                      int d, int f, int accumulate, T* __restrict__ dWd) {
  __shared__ float sA[TK][TM], sB[TK][TN];
  const int e = blockIdx.z, c0 = blockIdx.y * TM, i0 = blockIdx.x * TN;
  const int p0 = off[e], K = off[e + 1] - off[e];
  auto a_at = [&](int m, int k) -> float {
    return c0 + m < d ? to_f(dy[(size_t)row_token[p0 + k] * d + c0 + m]) : 0.f;
  };
  auto b_at = [&](int k, int n) -> float { return to_f(hg[(size_t)(p0 + k) * f + i0 + n]); };
  float acc[4][4] = {};
  tile_mma(a_at, b_at, K, acc, sA, sB);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = c0 + ty * 4 + i;
    if (c >= d) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      T& o = dWd[((size_t)e * d + c) * f + i0 + tx * 4 + j];
      o = from_f<T>(accumulate ? acc[i][j] + to_f(o) : acc[i][j]);
    }
  }
}

inline int max_tiles64(const Layer& L, const Bufs& B) { return 2 * ((B.R + kBM - 1) / kBM + L.E + L.S); }

}  // namespace

#define MOE_DISPATCH(L, ...)                         \
  do {                                               \
    if ((L).prec == MOE_FP32) {                      \
      typedef float T;                               \
      __VA_ARGS__;                                   \
    } else {                                         \
      typedef bf16 T;                                \
      __VA_ARGS__;                                   \
    }                                                \
  } while (0)

cudaError_t launch_simt_gateup(const Layer& L, const Bufs& B, const void* x, cudaStream_t s) {
  dim3 grid(max_tiles64(L, B), L.f / 32);
  MOE_DISPATCH(L, gateup_kernel<T><<<grid, 256, 0, s>>>((const T*)x, (const T*)L.W13, B.off, B.mt_off, B.row_token,
                                                        L.E + L.S, L.d, L.f, L.G, (T*)B.h, (T*)B.uv));
  return cudaGetLastError();
}

cudaError_t launch_simt_down(const Layer& L, const Bufs& B, cudaStream_t s) {
  dim3 grid(max_tiles64(L, B), (L.d + TN - 1) / TN);
  MOE_DISPATCH(L, down_kernel<T><<<grid, 256, 0, s>>>((const T*)B.h, (const T*)L.Wd, B.off, B.mt_off, B.row_gate,
                                                      L.E + L.S, L.d, L.f, (T*)B.o));
  return cudaGetLastError();
}

cudaError_t launch_simt_bwd_dh(const Layer& L, const Bufs& B, const void* dy, cudaStream_t s) {
  dim3 grid(max_tiles64(L, B), L.f / TN);
  MOE_DISPATCH(L, bwd_dh_kernel<T><<<grid, 256, 0, s>>>((const T*)dy, (const T*)L.Wd, (const T*)B.uv, B.off,
                                                        B.mt_off, B.row_token, B.row_gate, L.E + L.S, B.A, L.d, L.f,
                                                        L.G, (T*)B.dudv, (T*)B.hg, B.dg_part));
  return cudaGetLastError();
}

cudaError_t launch_simt_bwd_dx(const Layer& L, const Bufs& B, cudaStream_t s) {
  dim3 grid(max_tiles64(L, B), (L.d + TN - 1) / TN);
  MOE_DISPATCH(L, bwd_dx_kernel<T><<<grid, 256, 0, s>>>((const T*)B.dudv, (const T*)L.W13, B.off, B.mt_off,
                                                        L.E + L.S, L.d, L.f, (T*)B.dx_rows));
  return cudaGetLastError();
}

cudaError_t launch_simt_bwd_dw13(const Layer& L, const Bufs& B, const void* x, void* dWg, void* dWu, bool acc,
                                cudaStream_t s) {
  dim3 g13((L.d + TN - 1) / TN, 2 * L.f / TM, L.E + L.S);
  MOE_DISPATCH(L, bwd_dw13_kernel<T><<<g13, 256, 0, s>>>((const T*)B.dudv, (const T*)x, B.off, B.row_token, L.d, L.f,
                                                         L.G, acc ? 1 : 0, (T*)dWg, (T*)dWu));
  return cudaGetLastError();
}

cudaError_t launch_simt_bwd_dwd(const Layer& L, const Bufs& B, const void* dy, void* dWd, bool acc, cudaStream_t s) {
  dim3 gd(L.f / TN, (L.d + TM - 1) / TM, L.E + L.S);
  MOE_DISPATCH(L, bwd_dwd_kernel<T><<<gd, 256, 0, s>>>((const T*)dy, (const T*)B.hg, B.off, B.row_token, L.d, L.f,
                                                       acc ? 1 : 0, (T*)dWd));
  return cudaGetLastError();
}

}  // namespace moe
