// Weighted combine, backward gather-sums, router backward and weight packing.
//
// The combine follows "Cursor открыл код ядра Mixture of Experts ..."
// (dzen.guru), section "Три решения, которые дали результат": results go back
// to the token that owns them, and the whole call is deterministic. Here every
// output element is one fp32 sum in a fixed order (shared expert first, then
// slots j = 0..k-1), with no floating-point atomics.
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace moe {

namespace {

// y[t, c] = o[A + t, c] (shared) + sum_j o[inv[t*k + j], c]. o already carries the gate.
// One thread per 8 (bf16) or 4 (fp32) consecutive columns.
template <typename T>
__global__ void __launch_bounds__(256) combine_kernel(const T* __restrict__ o, const int* __restrict__ inv, int Tn,
                                                      int d, int k, int A, int S, T* __restrict__ y) {
  griddep_wait();    // after the predecessor grid (launch.cuh)
  griddep_launch();
  constexpr int V = 16 / sizeof(T);
  const int vecs = d / V;
  const long q = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (q >= (long)Tn * vecs) return;
  const int t = (int)(q / vecs), c = (int)(q % vecs) * V;
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  auto add_row = [&](const uint4& u) {
    if constexpr (sizeof(T) == 2) {
      float f[8];
      unpack8(u, f);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += f[i];
    } else {
      acc[0] += __uint_as_float(u.x);
      acc[1] += __uint_as_float(u.y);
      acc[2] += __uint_as_float(u.z);
      acc[3] += __uint_as_float(u.w);
    }
  };
  // every row's load goes out before the first add (the sum keeps its order: shared, then j)
  int rows[kMaxK];
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) rows[j] = j < k ? inv[(long)t * k + j] : 0;
  uint4 v[kMaxK + 1];
  if (S) v[kMaxK] = *reinterpret_cast<const uint4*>(o + (long)(A + t) * d + c);
#pragma unroll
  for (int j = 0; j < kMaxK; ++j)
    if (j < k) v[j] = *reinterpret_cast<const uint4*>(o + (long)rows[j] * d + c);
  if (S) add_row(v[kMaxK]);
#pragma unroll
  for (int j = 0; j < kMaxK; ++j)
    if (j < k) add_row(v[j]);
  uint4 out;
  if constexpr (sizeof(T) == 2) {
    out = pack8(acc);
  } else {
    out = make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]), __float_as_uint(acc[2]),
                     __float_as_uint(acc[3]));
  }
  *reinterpret_cast<uint4*>(y + (long)t * d + c) = out;
}

// Gate gradient and router logit gradient, one warp per token.
// dg[t, j] = sum over the f/64 partials of sorted row inv[t*k + j], in order.
// Then dl per router kind (selected experts only when renormalised; every
// expert for a plain softmax): see the oracle's router_grad for the formulas.
__global__ void __launch_bounds__(256) router_dl_kernel(const float* __restrict__ logits, const int* __restrict__ idx,
                                                        const float* __restrict__ gate, const int* __restrict__ inv,
                                                        const float* __restrict__ dg_part, int nslots, int Tn, int E,
                                                        int k, int router, int renorm, float scale,
                                                        float* __restrict__ dgate, float* __restrict__ dl) {
  griddep_wait();    // after the predecessor grid (launch.cuh)
  griddep_launch();
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= Tn) return;
  float dg[kMaxK], g[kMaxK], l[kMaxK];
  int ex[kMaxK];
  float dot = 0.f;
  // lane j sums slot j's partials (in order; their loads batched), then every lane takes all k
  float own = 0.f;
  if (lane < k) {
    const float* dp = dg_part + (long)inv[(long)t * k + lane] * nslots;
#pragma unroll 8
    for (int q = 0; q < nslots; ++q) own += dp[q];
  }
  for (int j = 0; j < k; ++j) {
    dg[j] = __shfl_sync(0xffffffffu, own, j);
    g[j] = gate[(long)t * k + j];
    ex[j] = idx[(long)t * k + j];
    l[j] = logits[(long)t * E + ex[j]];
    dot += g[j] * dg[j];
  }
  if (lane < k) {
    for (int j = 0; j < k; ++j)
      if (j == lane) dgate[(long)t * k + j] = dg[j];
  }
  float* dlr = dl + (long)t * E;
  if (router == MOE_ROUTER_SOFTMAX) {
    // g = scale * p: dl = p (scale*dg - sum_j p_j scale dg_j) on the selected set (renorm)
    // or on all experts with dg = 0 off the selection (plain softmax).
    const float dots = dot;  // sum_j g_j dg_j = scale * sum_j p_j dg_j
    if (renorm) {
      for (int e = lane; e < E; e += 32) dlr[e] = 0.f;
      __syncwarp();
      if (lane == 0)
        for (int j = 0; j < k; ++j) dlr[ex[j]] = (g[j] / scale) * (scale * dg[j] - dots);
    } else {
      float m = -INFINITY;
      for (int e = lane; e < E; e += 32) m = fmaxf(m, logits[(long)t * E + e]);
#pragma unroll
      for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float den = 0.f;
      for (int e = lane; e < E; e += 32) den += expf(logits[(long)t * E + e] - m);
      den = warp_sum(den);
      for (int e = lane; e < E; e += 32) {
        float dge = 0.f;
        for (int j = 0; j < k; ++j)
          if (ex[j] == e) dge = dg[j];
        const float p = expf(logits[(long)t * E + e] - m) / den;
        dlr[e] = p * (scale * dge - dots);
      }
    }
  } else {
    float S = 0.f;
    float s[kMaxK];
    for (int j = 0; j < k; ++j) {
      s[j] = 1.0f / (1.0f + expf(-l[j]));
      S += s[j];
    }
    for (int e = lane; e < E; e += 32) dlr[e] = 0.f;
    __syncwarp();
    if (lane == 0)
      for (int j = 0; j < k; ++j) {
        const float ds = renorm ? (scale / S) * (dg[j] - dot / scale) : scale * dg[j];
        dlr[ex[j]] = ds * s[j] * (1.f - s[j]);
      }
  }
}

// Renormalised routers: dl is nonzero only at the selected experts, so dWr[e] = sum over the
// segment's rows p of dl[t_p, e] x[t_p]. A segment of cnt rows is split ns = min(kRouterSplit,
// ceil(cnt / kRouterSplitRows)) ways, so a hot expert (thousands of rows) spreads over more SMs
// while ordinary ones stay whole. Block (column block, e, split s < ns) takes the rows
// p = off[e] + s + ns * (w + 8 i) of its warp w, each lane 16 bytes of columns; the 8 warp partials
// are added in warp order. With one split the block writes dWr[e] itself; otherwise it writes
// part[s][e] and router_dw_reduce_kernel adds the splits in order.
__device__ __forceinline__ int router_splits(int cnt) {
  const int ns = (cnt + kRouterSplitRows - 1) / kRouterSplitRows;
  return ns < 1 ? 1 : (ns > kRouterSplit ? kRouterSplit : ns);
}

template <typename T>
__global__ void __launch_bounds__(256) router_dw_seg_kernel(const float* __restrict__ dl, const T* __restrict__ x,
                                                            const int* __restrict__ off, const int* __restrict__ perm,
                                                            int d, int E, int k, int accumulate,
                                                            float* __restrict__ dWr, float* __restrict__ part) {
  griddep_wait();    // after the predecessor grid (launch.cuh)
  griddep_launch();
  constexpr int V = 16 / sizeof(T);
  __shared__ float red[8][32 * V];
  const int e = blockIdx.y, sp = blockIdx.z, lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int p0 = off[e], p1 = off[e + 1];
  const int ns = router_splits(p1 - p0);
  if (sp >= ns) return;
  const int c = blockIdx.x * 32 * V + lane * V;
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  if (c < d) {
#pragma unroll 8
    for (int p = p0 + sp + ns * w; p < p1; p += ns * 8) {
      const int t = perm[p] / k;
      const float g = dl[(long)t * E + e];
      const uint4 u = *reinterpret_cast<const uint4*>(x + (long)t * d + c);
      if constexpr (sizeof(T) == 2) {
        float f[8];
        unpack8(u, f);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(g, f[i], acc[i]);
      } else {
        acc[0] = fmaf(g, __uint_as_float(u.x), acc[0]);
        acc[1] = fmaf(g, __uint_as_float(u.y), acc[1]);
        acc[2] = fmaf(g, __uint_as_float(u.z), acc[2]);
        acc[3] = fmaf(g, __uint_as_float(u.w), acc[3]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < V; ++i) red[w][lane * V + i] = acc[i];
  __syncthreads();
  const int col = blockIdx.x * 32 * V + threadIdx.x;
  if (threadIdx.x < 32 * V && col < d) {
    float sum = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) sum += red[q][threadIdx.x];
    const long o = (long)e * d + col;
    if (ns == 1) dWr[o] = accumulate ? dWr[o] + sum : sum;
    else part[(long)sp * E * d + o] = sum;
  }
}

// Split segments: dWr[e] = (dWr[e] if accumulating) + sum over their splits s = 0 .. ns-1, in order.
__global__ void __launch_bounds__(256) router_dw_reduce_kernel(const float* __restrict__ part,
                                                               const int* __restrict__ off, int E, int d,
                                                               int accumulate, float* __restrict__ dWr) {
  griddep_wait();    // after the predecessor grid (launch.cuh)
  griddep_launch();
  const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  const long n = (long)E * d;
  if (i >= n) return;
  const int e = (int)(i / d);
  const int ns = router_splits(off[e + 1] - off[e]);
  if (ns == 1) return;
  float sum = 0.f;
  for (int sp = 0; sp < ns; ++sp) sum += part[sp * n + i];
  dWr[i] = accumulate ? dWr[i] + sum : sum;
}

// Plain softmax: dl is dense; dWr[e, c] over all tokens in order, one thread per (e, column).
template <typename T>
__global__ void __launch_bounds__(256) router_dw_dense_kernel(const float* __restrict__ dl, const T* __restrict__ x,
                                                              int Tn, int d, int E, int accumulate,
                                                              float* __restrict__ dWr) {
  griddep_wait();    // after the predecessor grid (launch.cuh)
  griddep_launch();
  const int e = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= d) return;
  float acc = 0.f;
  for (int t = 0; t < Tn; ++t) acc = fmaf(dl[(long)t * E + e], to_f(x[(long)t * d + c]), acc);
  dWr[(long)e * d + c] = accumulate ? dWr[(long)e * d + c] + acc : acc;
}

// dx[t, c] = dx_rows[A + t, c] (shared) + sum_j dx_rows[inv[t*k + j], c] + sum_e dl[t, e] Wr[e, c]
// (selected experts in slot order when renormalised, all experts otherwise).
// One thread per 16 bytes of a token row; fp32 sum in that fixed order.
template <typename T>
__global__ void __launch_bounds__(256) dx_gather_kernel(const T* __restrict__ dx_rows, const int* __restrict__ inv,
                                                        const int* __restrict__ idx, const float* __restrict__ dl,
                                                        const T* __restrict__ Wr, int Tn, int d, int E, int k, int A,
                                                        int S, int dense, T* __restrict__ dx) {
  griddep_wait();    // after the predecessor grid (launch.cuh)
  griddep_launch();
  constexpr int V = 16 / sizeof(T);
  const int vecs = d / V;
  const long q = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (q >= (long)Tn * vecs) return;
  const int t = (int)(q / vecs), c = (int)(q % vecs) * V;
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  auto add = [&](const T* src, float g) {
    const uint4 u = *reinterpret_cast<const uint4*>(src);
    if constexpr (sizeof(T) == 2) {
      float f[8];
      unpack8(u, f);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(g, f[i], acc[i]);
    } else {
      acc[0] = fmaf(g, __uint_as_float(u.x), acc[0]);
      acc[1] = fmaf(g, __uint_as_float(u.y), acc[1]);
      acc[2] = fmaf(g, __uint_as_float(u.z), acc[2]);
      acc[3] = fmaf(g, __uint_as_float(u.w), acc[3]);
    }
  };
  if (S) add(dx_rows + (long)(A + t) * d + c, 1.f);
  for (int j = 0; j < k; ++j) add(dx_rows + (long)inv[(long)t * k + j] * d + c, 1.f);
  if (dense) {
    for (int e = 0; e < E; ++e) add(Wr + (long)e * d + c, dl[(long)t * E + e]);
  } else {
    for (int j = 0; j < k; ++j) {
      const int e = idx[(long)t * k + j];
      add(Wr + (long)e * d + c, dl[(long)t * E + e]);
    }
  }
  uint4 out;
  if constexpr (sizeof(T) == 2) {
    out = pack8(acc);
  } else {
    out = make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]), __float_as_uint(acc[2]),
                     __float_as_uint(acc[3]));
  }
  *reinterpret_cast<uint4*>(dx + (long)t * d + c) = out;
}

// Packing: W13 rows interleave gate and up in blocks of G rows; Wd, Wr, bias are copied.
template <typename T>
__global__ void pack_w13_kernel(const T* __restrict__ Wg, const T* __restrict__ Wu, int nseg, int f, int d, int G,
                                T* __restrict__ W13) {
  const long row = blockIdx.x;          // packed row over all experts
  const int e = (int)(row / (2 * f)), pr = (int)(row % (2 * f));
  const int blk = pr / (2 * G), w = pr % (2 * G);
  const int feat = blk * G + (w % G);
  const T* src = (w < G ? Wg : Wu) + ((long)e * f + feat) * d;
  T* dst = W13 + row * d;
  for (int c = threadIdx.x; c < d; c += blockDim.x) dst[c] = src[c];
}

}  // namespace

cudaError_t launch_combine(const Layer& L, const Bufs& B, void* y, cudaStream_t s) {
  const int V = 16 / (int)elem_bytes(L.prec);
  const long n = (long)B.T * (L.d / V);
  const int blocks = (int)((n + 255) / 256);
  if (L.prec == MOE_FP32)
    MOE_TRY(launch_pdl(combine_kernel<float>, dim3(blocks), dim3(256), 0, s, (const float*)B.o, B.inv, B.T, L.d, L.k,
        B.A, L.S, (float*)y));
  else
    MOE_TRY(launch_pdl(combine_kernel<bf16>, dim3(blocks), dim3(256), 0, s, (const bf16*)B.o, B.inv, B.T, L.d, L.k,
        B.A, L.S, (bf16*)y));
  return cudaGetLastError();
}

cudaError_t launch_router_bwd(const Layer& L, const Bufs& B, const void* x, float* dWr, bool acc, cudaStream_t s) {
  const int dense = (L.router == MOE_ROUTER_SOFTMAX && !L.renorm) ? 1 : 0;
  MOE_TRY(launch_pdl(router_dl_kernel, dim3((B.T * 32 + 255) / 256), dim3(256), 0, s, B.logits, B.idx, B.gate, B.inv,
      B.dg_part, L.f / 64, B.T, L.E, L.k, L.router, L.renorm, L.scale, B.dgate, B.dl));
  if (dense) {
    dim3 grid((L.d + 255) / 256, L.E);
    if (L.prec == MOE_FP32)
      MOE_TRY(launch_pdl(router_dw_dense_kernel<float>, dim3(grid), dim3(256), 0, s, B.dl, (const float*)x, B.T, L.d,
          L.E, acc, dWr));
    else
      MOE_TRY(launch_pdl(router_dw_dense_kernel<bf16>, dim3(grid), dim3(256), 0, s, B.dl, (const bf16*)x, B.T, L.d,
          L.E, acc, dWr));
  } else {
    const int cols = 32 * 16 / (int)elem_bytes(L.prec);
    dim3 grid((L.d + cols - 1) / cols, L.E, kRouterSplit);
    if (L.prec == MOE_FP32)
      MOE_TRY(launch_pdl(router_dw_seg_kernel<float>, dim3(grid), dim3(256), 0, s, B.dl, (const float*)x, B.off,
          B.perm, L.d, L.E, L.k, acc, dWr, B.dwr_part));
    else
      MOE_TRY(launch_pdl(router_dw_seg_kernel<bf16>, dim3(grid), dim3(256), 0, s, B.dl, (const bf16*)x, B.off, B.perm,
          L.d, L.E, L.k, acc, dWr, B.dwr_part));
    const long n = (long)L.E * L.d;
    MOE_TRY(launch_pdl(router_dw_reduce_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, B.dwr_part, B.off,
        L.E, L.d, acc, dWr));
  }
  return cudaGetLastError();
}

cudaError_t launch_dx_gather(const Layer& L, const Bufs& B, void* dx, cudaStream_t s) {
  const int dense = (L.router == MOE_ROUTER_SOFTMAX && !L.renorm) ? 1 : 0;
  const int V = 16 / (int)elem_bytes(L.prec);
  const long n = (long)B.T * (L.d / V);
  const int blocks = (int)((n + 255) / 256);
  if (L.prec == MOE_FP32)
    MOE_TRY(launch_pdl(dx_gather_kernel<float>, dim3(blocks), dim3(256), 0, s, (const float*)B.dx_rows, B.inv, B.idx,
        B.dl, (const float*)L.Wr, B.T, L.d, L.E, L.k, B.A, L.S, dense, (float*)dx));
  else
    MOE_TRY(launch_pdl(dx_gather_kernel<bf16>, dim3(blocks), dim3(256), 0, s, (const bf16*)B.dx_rows, B.inv, B.idx,
        B.dl, (const bf16*)L.Wr, B.T, L.d, L.E, L.k, B.A, L.S, dense, (bf16*)dx));
  return cudaGetLastError();
}

cudaError_t launch_pack_weights(const Layer& L, const void* Wr, const float* bias, const void* Wg, const void* Wu,
                                const void* Wd, cudaStream_t s) {
  const size_t eb = elem_bytes(L.prec);
  const int nseg = L.E + L.S;
  const long rows = (long)nseg * 2 * L.f;
  if (L.prec == MOE_FP32)
    pack_w13_kernel<float><<<rows, 256, 0, s>>>((const float*)Wg, (const float*)Wu, nseg, L.f, L.d, L.G,
                                                (float*)L.W13);
  else
    pack_w13_kernel<bf16><<<rows, 256, 0, s>>>((const bf16*)Wg, (const bf16*)Wu, nseg, L.f, L.d, L.G, (bf16*)L.W13);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  err = cudaMemcpyAsync(L.Wd, Wd, (size_t)nseg * L.d * L.f * eb, cudaMemcpyDeviceToDevice, s);
  if (err != cudaSuccess) return err;
  err = cudaMemcpyAsync(L.Wr, Wr, (size_t)L.E * L.d * eb, cudaMemcpyDeviceToDevice, s);
  if (err != cudaSuccess) return err;
  if (bias) return cudaMemcpyAsync(L.bias, bias, (size_t)L.E * sizeof(float), cudaMemcpyDeviceToDevice, s);
  return cudaMemsetAsync(L.bias, 0, (size_t)L.E * sizeof(float), s);
}

}  // namespace moe
