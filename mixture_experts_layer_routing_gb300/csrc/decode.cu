// Small-batch decode with one output value per warp.
//
// Follows "Cursor a réécrit le décodage de MoE" (toolnavs.com): in section
// "Cursor a réécrit le décodage de MoE" the parallel axis is flipped from
// experts to outputs, each warp owning one output value, for small batches;
// in section "1.84x plus de vitesse ..." the whole MoE layer runs in two
// kernels, without multi-step staging, cross-warp synchronisation or extra
// buffers, and the output sits closer to an FP32 reference.
// Here:
//   route     one to eight warps per (token, expert) router logit (split along d
//             when B x E is small, so that every SM streams part of Wr; the
//             partial sums are added in warp order); then one block (launched
//             ahead, programmatic dependent launch) selects the top-k of every
//             token and lists the used experts U (ascending, the shared expert
//             last) with their tokens.
//   gate/up   warp per (expert in U, row i): streams Wg[e][i,:] and Wu[e][i,:]
//             once with 16-byte coalesced loads and produces h[t, slot, i] =
//             silu(u) v in fp32 for every token routed to e.
//   down      warp per two (bf16) or three (MXFP8) output columns c: for each
//             e in U ascending, streams Wd[e][c,:] once and adds gate * (h . w)
//             to each token's fp32 accumulator; y[:, c] is written once. No
//             atomics.
// Intermediates stay fp32 (h is never rounded to bf16). The kernels are bound
// by the weight bytes each warp keeps in flight, so a single-token batch runs
// shapes that spend the registers of a token group on deeper load batches.
//
// MXFP8 layers decode the same way on their E4M3 weights (one E8M0 scale per
// 32 values along each product's K): x is quantised along d and h along f
// before the down projection, as the MXFP8 layer forward does, so decode is
// that forward on B tokens. The weight bytes per expert halve.
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "mx_quant.cuh"
#include "topk.cuh"
#include "launch.cuh"

namespace moe {

namespace {

struct DecodeWs {
  float* logits;   // [B, E]
  int* nU;         // [1]
  int* U;          // [E + 1]   experts in use, ascending, shared expert (E) last
  int* u_off;      // [E + 2]   token-list offsets per U entry
  int* a_tok;      // [B*k + B] (t << 8) | slot
  float* a_gate;   // [B*k + B]
  float* h;        // [B, k+1, f]
  // MXFP8 layers only: the quantised activations as their E4M3 codes held in fp16 (every E4M3
  // value is exact in fp16) and one E8M0 byte per 32 values; value = code * 2^(scale - 127).
  uint16_t* xc;    // [B, d]      x quantised along d: codes
  uint8_t* xs;     // [B, d/32]   and scales
  uint16_t* hc;    // [B, k+1, f] h quantised along f: codes
  uint8_t* hs;     // [B, k+1, f/32]
};

inline size_t al(size_t v) { return (v + 255) & ~size_t(255); }

DecodeWs carve(const Layer& L, int B, void* ws) {
  char* p = (char*)ws;
  DecodeWs w;
  const int na = B * L.k + B;
  w.logits = (float*)p; p += al(sizeof(float) * B * L.E);
  w.nU = (int*)p; p += al(sizeof(int));
  w.U = (int*)p; p += al(sizeof(int) * (L.E + 1));
  w.u_off = (int*)p; p += al(sizeof(int) * (L.E + 2));
  w.a_tok = (int*)p; p += al(sizeof(int) * na);
  w.a_gate = (float*)p; p += al(sizeof(float) * na);
  w.h = (float*)p; p += al(sizeof(float) * B * (L.k + 1) * L.f);
  w.xc = w.hc = nullptr;
  w.xs = w.hs = nullptr;
  if (L.prec == MOE_MXFP8) {
    w.xc = (uint16_t*)p; p += al(2 * (size_t)B * L.d);
    w.xs = (uint8_t*)p; p += al((size_t)B * L.d / 32);
    w.hc = (uint16_t*)p; p += al(2 * (size_t)B * (L.k + 1) * L.f);
    w.hs = (uint8_t*)p; p += al((size_t)B * (L.k + 1) * L.f / 32);
  }
  return w;
}

// 32 fp32 values -> their MX quantisation: 32 E4M3 codes written as fp16 values (64 bytes at
// codes), the E8M0 byte at *scale.
__device__ __forceinline__ void quant32_to_f16(const float (&v)[32], uint16_t* codes, uint8_t* scale) {
  uint4 q[2];
  *scale = quant32(v, q[0], q[1]);
  uint4* dst = reinterpret_cast<uint4*>(codes);
#pragma unroll
  for (int hlf = 0; hlf < 2; ++hlf) {
    const uint32_t w[4] = {q[hlf].x, q[hlf].y, q[hlf].z, q[hlf].w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] & 0xffffu), __NV_E4M3);
      const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] >> 16), __NV_E4M3);
      o[2 * i] = (uint32_t)lo.x | ((uint32_t)lo.y << 16);
      o[2 * i + 1] = (uint32_t)hi.x | ((uint32_t)hi.y << 16);
    }
    dst[2 * hlf] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[2 * hlf + 1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// x [B, d] bf16 -> xc, xs (MXFP8 layers), 32-value block b.
__device__ __forceinline__ void quant_x_block(const bf16* __restrict__ x, int b, const DecodeWs& w) {
  float v[32];
#pragma unroll
  for (int q = 0; q < 4; ++q) unpack8(*reinterpret_cast<const uint4*>(x + (size_t)b * 32 + 8 * q), v + 8 * q);
  quant32_to_f16(v, w.xc + (size_t)b * 32, w.xs + b);
}

constexpr int kRouteWarps = 8;
constexpr int kBatch = 7;   // 16-byte chunks per lane loaded before they are used

__global__ void __launch_bounds__(kRouteWarps * 32) decode_logits_kernel(const bf16* __restrict__ x,
                                                                       const bf16* __restrict__ Wr, int B, int d,
                                                                       int E, int parts, DecodeWs w, int quant_x) {
  griddep_launch();
  // MXFP8 layers: the blocks also quantise x along d for the gate/up kernel (one launch fewer)
  if (quant_x)
    for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < B * d / 32; b += gridDim.x * blockDim.x) quant_x_block(x, b, w);
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  // `parts` consecutive warps of a block share one (t, e); warp `part` takes the 16-byte chunks
  // part*32 + lane, + 32*parts, ...
  const int item = blockIdx.x * (kRouteWarps / parts) + wib / parts, part = wib % parts;
  __shared__ float red[kRouteWarps];
  float acc = 0.f;
  if (item < B * E) {
    const int t = item / E, e = item % E;
    const bf16* xr = x + (size_t)t * d;
    const bf16* wr = Wr + (size_t)e * d;
    const int nchunk = d / 8, step = 32 * parts;
    for (int cb = part * 32 + lane; cb < nchunk; cb += step * kBatch) {
      uint4 wv[kBatch], xv[kBatch];
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const int c = cb + q * step;
        if (c < nchunk) {
          wv[q] = ld_stream(wr + c * 8);
          xv[q] = *reinterpret_cast<const uint4*>(xr + c * 8);
        }
      }
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        if (cb + q * step < nchunk) {
          float a[8], b[8];
          unpack8(xv[q], a);
          unpack8(wv[q], b);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc = fmaf(a[i], b[i], acc);
        }
      }
    }
    acc = warp_sum(acc);
  }
  if (lane == 0) red[wib] = acc;
  __syncthreads();
  if (item < B * E && part == 0 && lane == 0) {
    float sum = red[wib];
    for (int q = 1; q < parts; ++q) sum += red[wib + q];
    w.logits[item] = sum;
  }
}

// One block: selects the top-k of every token from the logits and lists the used experts U
// (ascending, the shared expert last) with their tokens. Launched after decode_logits_kernel with
// programmatic dependent launch, so it is resident before the logits are complete and starts when
// they are.
__global__ void __launch_bounds__(kRouteWarps * 32) decode_select_kernel(const float* __restrict__ bias, int B, int E,
                                                                       int k, int S, int router, int renorm,
                                                                       float scale, DecodeWs w) {
  griddep_launch();
  griddep_wait();
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  // the selection stays in shared memory: only this block reads it
  __shared__ int s_idx[kMaxDecodeB * kMaxK];
  __shared__ float s_gate[kMaxDecodeB * kMaxK];
  for (int t = wib; t < B; t += kRouteWarps)
    warp_topk_gates(w.logits + (size_t)t * E, bias, E, k, router, renorm, scale, s_idx + t * k, s_gate + t * k);
  __syncthreads();
  // experts in use and their token lists (stable: ascending assignment); thread e owns expert e
  __shared__ int cnt[kMaxE + 1];
  __shared__ int start[kMaxE + 2];
  __shared__ int wsum[kRouteWarps][2];
  for (int e = threadIdx.x; e <= E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int A = B * k;
  for (int a = threadIdx.x; a < A; a += blockDim.x) atomicAdd(&cnt[s_idx[a]], 1);
  __syncthreads();
  {
    // block-wide exclusive scans of (expert used, its count) over e = threadIdx.x < E
    const int e = threadIdx.x;
    const int c = e < E ? cnt[e] : 0;
    int used = c > 0 ? 1 : 0, run = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int nu = __shfl_up_sync(0xffffffffu, used, o), nr = __shfl_up_sync(0xffffffffu, run, o);
      if (lane >= o) {
        used += nu;
        run += nr;
      }
    }
    if (lane == 31) {
      wsum[wib][0] = used;
      wsum[wib][1] = run;
    }
    __syncthreads();
    int bu = 0, br = 0;
    for (int q = 0; q < wib; ++q) {
      bu += wsum[q][0];
      br += wsum[q][1];
    }
    int totu = 0, totr = 0;
    for (int q = 0; q < kRouteWarps; ++q) {
      totu += wsum[q][0];
      totr += wsum[q][1];
    }
    const int pos_u = bu + used - (c > 0 ? 1 : 0), pos_r = br + run - c;
    if (c > 0) {
      start[e] = pos_r;
      w.U[pos_u] = e;
      w.u_off[pos_u] = pos_r;
    }
    if (threadIdx.x == 0) {
      int nU = totu, r0 = totr;
      if (S) {
        start[E] = r0;
        w.U[nU] = E;
        w.u_off[nU] = r0;
        r0 += B;
        ++nU;
      }
      w.u_off[nU] = r0;
      *w.nU = nU;
    }
  }
  __syncthreads();
  for (int a = threadIdx.x; a < A; a += blockDim.x) {
    const int e = s_idx[a];
    int rank = 0;
    for (int q = 0; q < a; ++q) rank += (s_idx[q] == e);
    const int pos = start[e] + rank;
    w.a_tok[pos] = ((a / k) << 8) | (a % k);
    w.a_gate[pos] = s_gate[a];
  }
  if (S)
    for (int t = threadIdx.x; t < B; t += blockDim.x) {
      w.a_tok[start[E] + t] = (t << 8) | k;
      w.a_gate[start[E] + t] = 1.0f;
    }
}


constexpr int kTokGroup = 4;

// One warp per (U entry, row i) item, grid-stride over items. Each lane loads
// NB 16-byte chunks of both weight rows before using any of them; TG tokens of
// the expert per pass. Launched as (kTokGroup, kBatch), and as (1, 10) for a
// single token, where the registers of the token group go to a deeper batch.
template <int TG, int NB>
__global__ void __launch_bounds__(256, 2) decode_gateup_kernel(const bf16* __restrict__ x, const bf16* __restrict__ W13,
                                                            int d, int f, int G, int k, int E, int S, DecodeWs w) {
  // The shared expert is used by every token whatever the routing: while the
  // router still runs, pull its gate/up rows into L2 (each block one slice).
  if (S && threadIdx.x == 0) {
    const size_t bytes = (size_t)2 * f * d * sizeof(bf16);
    const size_t slice = ((bytes + gridDim.x - 1) / gridDim.x + 15) & ~(size_t)15;
    const size_t b0 = (size_t)blockIdx.x * slice;
    if (b0 < bytes) {
      const char* base = (const char*)(W13 + (size_t)E * 2 * f * d) + b0;
      const size_t n = (bytes - b0) < slice ? (bytes - b0) : slice;
      for (size_t o = 0; o < n; o += 65536) {
        const uint32_t sz = (uint32_t)((n - o) < 65536 ? (n - o) : 65536);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(base + o), "r"(sz) : "memory");
      }
    }
  }
  griddep_wait();
  // the next kernel may launch once every block is past the routing (it reads the lists early)
  griddep_launch();
  const int lane = threadIdx.x & 31;
  const int nU = *w.nU;
  const int items = nU * f;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  const int nchunk = d / 8;
  for (int it = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); it < items; it += nwarps) {
    // the last U entry (the shared expert when there is one) first: its rows are already in L2
    const int ui = (it / f + nU - 1) % nU, i = it % f;
    const int e = w.U[ui];
    const int a0 = w.u_off[ui], a1 = w.u_off[ui + 1];
    const bf16* wg = W13 + ((size_t)e * 2 * f + (i / G) * 2 * G + (i % G)) * d;
    const bf16* wu = wg + (size_t)G * d;
    for (int g0 = a0; g0 < a1; g0 += TG) {
      const int nt = min(TG, a1 - g0);
      const bf16* xr[TG];
#pragma unroll
      for (int q = 0; q < TG; ++q) xr[q] = x + (size_t)(q < nt ? (w.a_tok[g0 + q] >> 8) : 0) * d;
      float au[TG], av[TG];
#pragma unroll
      for (int q = 0; q < TG; ++q) au[q] = av[q] = 0.f;
      for (int cb = lane; cb < nchunk; cb += 32 * NB) {
        uint4 gv[NB], uvv[NB];
#pragma unroll
        for (int q = 0; q < NB; ++q) {
          const int c = cb + q * 32;
          if (c < nchunk) {
            gv[q] = ld_stream(wg + c * 8);
            uvv[q] = ld_stream(wu + c * 8);
          }
        }
#pragma unroll
        for (int q = 0; q < NB; ++q) {
          const int c = cb + q * 32;
          if (c < nchunk) {
            float fg[8], fu[8];
            unpack8(gv[q], fg);
            unpack8(uvv[q], fu);
#pragma unroll
            for (int tt = 0; tt < TG; ++tt) {
              if (tt < nt) {
                float xv[8];
                unpack8(*reinterpret_cast<const uint4*>(xr[tt] + c * 8), xv);
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                  au[tt] = fmaf(xv[r], fg[r], au[tt]);
                  av[tt] = fmaf(xv[r], fu[r], av[tt]);
                }
              }
            }
          }
        }
      }
#pragma unroll
      for (int tt = 0; tt < TG; ++tt) {
        if (tt < nt) {
          const float u = warp_sum(au[tt]);
          const float v = warp_sum(av[tt]);
          if (lane == 0) {
            const int code = w.a_tok[g0 + tt];
            const int t = code >> 8, slot = code & 255;
            w.h[((size_t)t * (k + 1) + slot) * f + i] = silu_f(u) * v;
          }
        }
      }
    }
  }
}

constexpr int kCols = 2;       // output columns per warp in the down kernel
constexpr int kDownWarps = 8;
constexpr int kFChunks = 8;    // 16-byte chunks of a Wd row per lane (f <= 2048 per pass)

// Loads the Wd rows c0.. (kCols of them) of expert e, features [f0, f0 + 2048), into registers.
__device__ __forceinline__ void load_wd(const bf16* Wd, int e, int d, int f, int c0, int f0, int lane,
                                        uint4 (&wv)[kCols][kFChunks]) {
#pragma unroll
  for (int cc = 0; cc < kCols; ++cc) {
    const bf16* row = Wd + ((size_t)e * d + c0 + cc) * f + f0;
#pragma unroll
    for (int q = 0; q < kFChunks; ++q) {
      const int c = (lane + 32 * q) * 8;
      if (f0 + c < f) wv[cc][q] = ld_stream(row + c);
    }
  }
}

__global__ void __launch_bounds__(kDownWarps * 32) decode_down_kernel(const bf16* __restrict__ Wd, int B, int d, int f,
                                                                      int k, DecodeWs w, bf16* __restrict__ y) {
  extern __shared__ float acc_s[];   // [kDownWarps][B][kCols]
  griddep_launch();
  // The routing lists are complete once this grid runs (the gate/up kernel lets it launch only
  // after its own wait on the routing), so the first expert's rows go out before waiting for h.
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  float* acc = acc_s + (size_t)wib * B * kCols;
  const int nU = __ldcg(w.nU);
  const int c0 = (blockIdx.x * kDownWarps + wib) * kCols;
  if (c0 >= d) return;
  uint4 wcur[kCols][kFChunks], wnext[kCols][kFChunks];
  load_wd(Wd, __ldcg(w.U), d, f, c0, 0, lane, wnext);
  griddep_wait();
  for (int q = lane; q < B * kCols; q += 32) acc[q] = 0.f;
  __syncwarp();
  for (int f0 = 0; f0 < f; f0 += 32 * kFChunks * 8) {
    if (f0 > 0) load_wd(Wd, w.U[0], d, f, c0, f0, lane, wnext);
    for (int ui = 0; ui < nU; ++ui) {
#pragma unroll
      for (int cc = 0; cc < kCols; ++cc)
#pragma unroll
        for (int q = 0; q < kFChunks; ++q) wcur[cc][q] = wnext[cc][q];
      if (ui + 1 < nU) load_wd(Wd, w.U[ui + 1], d, f, c0, f0, lane, wnext);   // next expert in flight
      const int a0 = w.u_off[ui], a1 = w.u_off[ui + 1];
      for (int a = a0; a < a1; ++a) {
        const int code = w.a_tok[a];
        const int t = code >> 8, slot = code & 255;
        const float g = w.a_gate[a];
        const float* hr = w.h + ((size_t)t * (k + 1) + slot) * f + f0;
        float s[kCols] = {};
#pragma unroll
        for (int q = 0; q < kFChunks; ++q) {
          const int c = (lane + 32 * q) * 8;
          if (f0 + c < f) {
            const float4 h0 = *reinterpret_cast<const float4*>(hr + c);
            const float4 h1 = *reinterpret_cast<const float4*>(hr + c + 4);
            const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
            for (int cc = 0; cc < kCols; ++cc) {
              float wf[8];
              unpack8(wcur[cc][q], wf);
#pragma unroll
              for (int r = 0; r < 8; ++r) s[cc] = fmaf(hv[r], wf[r], s[cc]);
            }
          }
        }
#pragma unroll
        for (int cc = 0; cc < kCols; ++cc) {
          const float tot = warp_sum(s[cc]);
          if (lane == 0) acc[t * kCols + cc] = fmaf(g, tot, acc[t * kCols + cc]);
        }
        __syncwarp();
      }
    }
  }
  __syncwarp();
  for (int q = lane; q < B * kCols; q += 32) {
    const int t = q / kCols, cc = q % kCols;
    if (c0 + cc < d) y[(size_t)t * d + c0 + cc] = __float2bfloat16_rn(acc[q]);
  }
}

// ------------------------------------------------------------------ MXFP8
// 2^(s - 127) for an E8M0 byte s (s = 0 is the subnormal 2^-127).
__device__ __forceinline__ float e8m0(uint32_t s) {
  return s ? __uint_as_float(s << 23) : __uint_as_float(0x00400000u);
}


// acc + a * b for fp16 a, b (exact products) with fp32 accumulation, one rounding per step.
__device__ __forceinline__ float fma_h(uint32_t a, uint32_t b, float c) {
  float d;
  asm("fma.rn.f32.f16 %0, %1, %2, %3;" : "=f"(d) : "h"((unsigned short)a), "h"((unsigned short)b), "f"(c));
  return d;
}

// sum_{i < 16} w[i] * a[i] in order i = 0..15, fp32 accumulation: w = 16 E4M3 codes (one 16-byte
// chunk), a = 16 fp16 codes (two 16-byte chunks). The codes are exact in fp16, so every product is
// exact and only the running sum rounds.
__device__ __forceinline__ float dot16_codes(const uint4& w, const uint4& a0, const uint4& a1) {
  const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
  const uint32_t aa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
  float acc = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(ww[q] & 0xffffu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(ww[q] >> 16), __NV_E4M3);
    acc = fma_h(lo.x, aa[2 * q], acc);
    acc = fma_h(lo.y, aa[2 * q] >> 16, acc);
    acc = fma_h(hi.x, aa[2 * q + 1], acc);
    acc = fma_h(hi.y, aa[2 * q + 1] >> 16, acc);
  }
  return acc;
}


// Gate/up on E4M3 weights: one warp per (U entry, row i); each lane takes 16-byte chunks (16
// values, half of a 32-value scale block) of the gate and up rows, decodes them once and applies
// the block scale to each token's partial dot product.
// TG tokens of an expert per pass, NB 16-byte chunks per lane per row in flight; launched as (1, 7):
// one token per pass leaves the registers for seven chunks per row in flight at two blocks per SM
// (with four tokens per pass only four fit, and every B measured ran slower).
template <int TG, int NB>
__global__ void __launch_bounds__(256, 2) decode_gateup_mx_kernel(const uint8_t* __restrict__ W13q,
                                                               const uint8_t* __restrict__ W13s, int d, int f, int G,
                                                               int k, int E, int S, DecodeWs w) {
  if (S && threadIdx.x == 0) {   // the shared expert's rows into L2 while the router runs
    const size_t bytes = (size_t)2 * f * d;
    const size_t slice = ((bytes + gridDim.x - 1) / gridDim.x + 15) & ~(size_t)15;
    const size_t b0 = (size_t)blockIdx.x * slice;
    if (b0 < bytes) {
      const char* base = (const char*)(W13q + (size_t)E * 2 * f * d) + b0;
      const size_t n = (bytes - b0) < slice ? (bytes - b0) : slice;
      for (size_t o = 0; o < n; o += 65536) {
        const uint32_t sz = (uint32_t)((n - o) < 65536 ? (n - o) : 65536);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(base + o), "r"(sz) : "memory");
      }
    }
  }
  griddep_wait();
  // the next kernel may launch once every block is past the routing (it reads the lists early)
  griddep_launch();
  const int lane = threadIdx.x & 31;
  const int nU = *w.nU;
  const int items = nU * f;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  const int nchunk = d / 16, nb = d / 32;
  for (int it = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); it < items; it += nwarps) {
    const int ui = (it / f + nU - 1) % nU, i = it % f;
    const int e = w.U[ui];
    const int a0 = w.u_off[ui], a1 = w.u_off[ui + 1];
    const size_t rg = (size_t)e * 2 * f + (i / G) * 2 * G + (i % G), ru = rg + G;
    const uint8_t* wg = W13q + rg * d;
    const uint8_t* wu = W13q + ru * d;
    for (int g0 = a0; g0 < a1; g0 += TG) {
      const int nt = min(TG, a1 - g0);
      const uint16_t* xr[TG];
      const uint8_t* xsr[TG];
#pragma unroll
      for (int q = 0; q < TG; ++q) {
        const size_t t = q < nt ? (w.a_tok[g0 + q] >> 8) : 0;
        xr[q] = w.xc + t * d;
        xsr[q] = w.xs + t * nb;
      }
      float au[TG], av[TG];
#pragma unroll
      for (int q = 0; q < TG; ++q) au[q] = av[q] = 0.f;
      for (int cb = lane; cb < nchunk; cb += 32 * NB) {
        uint4 gv[NB], uvv[NB];
        uint32_t sgv[NB], suv[NB];
#pragma unroll
        for (int q = 0; q < NB; ++q) {
          const int c = cb + q * 32;
          if (c < nchunk) {
            gv[q] = ld_stream(reinterpret_cast<const bf16*>(wg + (size_t)c * 16));
            uvv[q] = ld_stream(reinterpret_cast<const bf16*>(wu + (size_t)c * 16));
            sgv[q] = W13s[atom_k(rg, c >> 1, d)];
            suv[q] = W13s[atom_k(ru, c >> 1, d)];
          }
        }
#pragma unroll
        for (int q = 0; q < NB; ++q) {
          const int c = cb + q * 32;
          if (c < nchunk) {
            const float s_g = e8m0(sgv[q]), s_u = e8m0(suv[q]);
#pragma unroll
            for (int tt = 0; tt < TG; ++tt) {
              if (tt < nt) {
                // weight codes times x codes, then the x block scale and the weight block scale
                const uint4* xv8 = reinterpret_cast<const uint4*>(xr[tt] + (size_t)c * 16);
                const uint4 xa = xv8[0], xb = xv8[1];
                const float s_x = e8m0(xsr[tt][c >> 1]);
                au[tt] = fmaf(dot16_codes(gv[q], xa, xb) * s_x, s_g, au[tt]);
                av[tt] = fmaf(dot16_codes(uvv[q], xa, xb) * s_x, s_u, av[tt]);
              }
            }
          }
        }
      }
#pragma unroll
      for (int tt = 0; tt < TG; ++tt) {
        if (tt < nt) {
          const float u = warp_sum(au[tt]);
          const float v = warp_sum(av[tt]);
          if (lane == 0) {
            const int code = w.a_tok[g0 + tt];
            const int t = code >> 8, slot = code & 255;
            w.h[((size_t)t * (k + 1) + slot) * f + i] = silu_f(u) * v;
          }
        }
      }
    }
  }
}

// h [B, k+1, f] fp32 -> its MX quantisation along f (hc, hs); one thread per 32-value block.
__global__ void __launch_bounds__(256) decode_quant_h_kernel(int nblocks, DecodeWs w) {
  griddep_launch();
  griddep_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= nblocks) return;
  float v[32];
  const float4* src = reinterpret_cast<const float4*>(w.h + (size_t)b * 32);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float4 t = src[q];
    v[4 * q] = t.x;
    v[4 * q + 1] = t.y;
    v[4 * q + 2] = t.z;
    v[4 * q + 3] = t.w;
  }
  quant32_to_f16(v, w.hc + (size_t)b * 32, w.hs + b);
}


// The Wd rows c0.. of expert e, features [f0, f0 + 2048), and their block scales (as 2^(s-127)).
template <int NC, int FC>
__device__ __forceinline__ void load_wd_mx(const uint8_t* Wdq, const uint8_t* Wds, int e, int d, int f, int c0, int f0,
                                           int lane, uint4 (&wv)[NC][FC], uint32_t (&sv)[NC][FC]) {
#pragma unroll
  for (int cc = 0; cc < NC; ++cc) {
    const size_t r = (size_t)e * d + min(c0 + cc, d - 1);   // columns past d: any row (not stored)
    const uint8_t* row = Wdq + r * f + f0;
#pragma unroll
    for (int q = 0; q < FC; ++q) {
      const int c = (lane + 32 * q) * 16;
      if (f0 + c < f) {
        wv[cc][q] = ld_stream(reinterpret_cast<const bf16*>(row + c));
        sv[cc][q] = Wds[atom_k(r, (f0 + c) >> 5, f)];
      }
    }
  }
}

// Down on E4M3 weights: warp per pair of output columns, as the bf16 kernel; h comes quantised
// (as exact fp32 values); each Wd chunk is decoded and scaled once per expert.
// NC output columns per warp, FC 16-byte chunks of a Wd row per lane per pass over f; launched as
// (3, 2): three columns per warp fit the whole projection in one wave of blocks (two columns took
// 1.5 waves), and two chunks keep the registers of both experts' rows in flight.
// STAGE: the block first quantises h [B, k+1, f] along f itself, into shared memory (codes held in
// fp16 and the scale bytes, exactly as the h quantiser kernel would store them), so that kernel is
// not launched and the per-expert reads of h come from shared memory; taken while the staged h
// leaves two blocks per SM (B <= 3 at DeepSeek-V3 shapes). The first expert's weight rows are
// already in flight meanwhile.
template <int NC, int FC, bool STAGE>
__global__ void __launch_bounds__(kDownWarps * 32) decode_down_mx_kernel(const uint8_t* __restrict__ Wdq,
                                                                         const uint8_t* __restrict__ Wds, int B, int d,
                                                                         int f, int k, DecodeWs w,
                                                                         bf16* __restrict__ y) {
  extern __shared__ __align__(16) float acc_s[];   // [kDownWarps][B][NC], then (STAGE) h codes and scales
  griddep_launch();
  // The routing lists are complete once this grid runs (its predecessors let it launch only after
  // their own waits on the routing), so the first expert's rows go out before waiting for h.
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  float* acc = acc_s + (size_t)wib * B * NC;
  const int nU = __ldcg(w.nU);
  const int c0 = (blockIdx.x * kDownWarps + wib) * NC;
  const int nb = f / 32;
  uint4 wcur[NC][FC], wnext[NC][FC];
  uint32_t scur[NC][FC], snext[NC][FC];
  if (c0 < d) load_wd_mx<NC, FC>(Wdq, Wds, __ldcg(w.U), d, f, c0, 0, lane, wnext, snext);
  griddep_wait();
  const uint16_t* hc = w.hc;
  const uint8_t* hs = w.hs;
  if (STAGE) {
    const int na = B * (k + 1);
    uint16_t* shc = reinterpret_cast<uint16_t*>(acc_s + ((kDownWarps * B * NC + 3) & ~3));   // 16-byte aligned
    uint8_t* shs = reinterpret_cast<uint8_t*>(shc + (size_t)na * f);
    for (int b = threadIdx.x; b < na * nb; b += blockDim.x) {
      float v[32];
      const float4* src = reinterpret_cast<const float4*>(w.h + (size_t)b * 32);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 t4 = src[q];
        v[4 * q] = t4.x;
        v[4 * q + 1] = t4.y;
        v[4 * q + 2] = t4.z;
        v[4 * q + 3] = t4.w;
      }
      quant32_to_f16(v, shc + (size_t)b * 32, shs + b);
    }
    __syncthreads();
    hc = shc;
    hs = shs;
  }
  if (c0 >= d) return;
  for (int q = lane; q < B * NC; q += 32) acc[q] = 0.f;
  __syncwarp();
  for (int f0 = 0; f0 < f; f0 += 32 * FC * 16) {
    if (f0 > 0) load_wd_mx<NC, FC>(Wdq, Wds, w.U[0], d, f, c0, f0, lane, wnext, snext);
    for (int ui = 0; ui < nU; ++ui) {
#pragma unroll
      for (int cc = 0; cc < NC; ++cc)
#pragma unroll
        for (int q = 0; q < FC; ++q) {
          wcur[cc][q] = wnext[cc][q];
          scur[cc][q] = snext[cc][q];
        }
      if (ui + 1 < nU) load_wd_mx<NC, FC>(Wdq, Wds, w.U[ui + 1], d, f, c0, f0, lane, wnext, snext);   // next expert in flight
      const int a0 = w.u_off[ui], a1 = w.u_off[ui + 1];
      if (a1 - a0 == 1) {
        // one token (the common case at small B): no decoded copy of the chunk is kept
        const int code = w.a_tok[a0];
        const int t = code >> 8, slot = code & 255;
        const float g = w.a_gate[a0];
        const size_t hrow = (size_t)t * (k + 1) + slot;
        const uint16_t* hr = hc + hrow * f;
        const uint8_t* hsr = hs + hrow * nb;
        float s[NC] = {};
#pragma unroll
        for (int q = 0; q < FC; ++q) {
          const int c = f0 + (lane + 32 * q) * 16;
          if (c < f) {
            const uint4 ha = *reinterpret_cast<const uint4*>(hr + c), hb = *reinterpret_cast<const uint4*>(hr + c + 8);
            const float s_h = e8m0(hsr[c >> 5]);
#pragma unroll
            for (int cc = 0; cc < NC; ++cc)
              s[cc] = fmaf(dot16_codes(wcur[cc][q], ha, hb) * s_h, e8m0(scur[cc][q]), s[cc]);
          }
        }
#pragma unroll
        for (int cc = 0; cc < NC; ++cc) {
          const float tot = warp_sum(s[cc]);
          if (lane == 0) acc[t * NC + cc] = fmaf(g, tot, acc[t * NC + cc]);
        }
        __syncwarp();
        continue;
      }
      // several tokens: in groups of kTokGroup, each chunk decoded and scaled once per group
      for (int g0 = a0; g0 < a1; g0 += kTokGroup) {
        const int nt = min(kTokGroup, a1 - g0);
        const uint16_t* hr[kTokGroup];
        const uint8_t* hsr[kTokGroup];
#pragma unroll
        for (int tt = 0; tt < kTokGroup; ++tt) {
          const int code = w.a_tok[g0 + (tt < nt ? tt : 0)];
          const size_t hrow = (size_t)(code >> 8) * (k + 1) + (code & 255);
          hr[tt] = hc + hrow * f;
          hsr[tt] = hs + hrow * nb;
        }
        float s[kTokGroup][NC] = {};
#pragma unroll
        for (int q = 0; q < FC; ++q) {
          const int c = f0 + (lane + 32 * q) * 16;
          if (c < f) {
#pragma unroll
            for (int tt = 0; tt < kTokGroup; ++tt) {
              if (tt < nt) {
                const uint4 ha = *reinterpret_cast<const uint4*>(hr[tt] + c);
                const uint4 hb = *reinterpret_cast<const uint4*>(hr[tt] + c + 8);
                const float s_h = e8m0(hsr[tt][c >> 5]);
#pragma unroll
                for (int cc = 0; cc < NC; ++cc)
                  s[tt][cc] = fmaf(dot16_codes(wcur[cc][q], ha, hb) * s_h, e8m0(scur[cc][q]), s[tt][cc]);
              }
            }
          }
        }
#pragma unroll
        for (int tt = 0; tt < kTokGroup; ++tt) {
          if (tt < nt) {
            const int code = w.a_tok[g0 + tt];
            const int t = code >> 8;
            const float g = w.a_gate[g0 + tt];
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) {
              const float tot = warp_sum(s[tt][cc]);
              if (lane == 0) acc[t * NC + cc] = fmaf(g, tot, acc[t * NC + cc]);
            }
          }
        }
        __syncwarp();
      }
    }
  }
  __syncwarp();
  for (int q = lane; q < B * NC; q += 32) {
    const int t = q / NC, cc = q % NC;
    if (c0 + cc < d) y[(size_t)t * d + c0 + cc] = __float2bfloat16_rn(acc[q]);
  }
}

// Launch with programmatic stream serialisation: the kernel may start while
// its predecessor finishes; it waits (griddepcontrol.wait) before reading the
// predecessor's results.

}  // namespace

size_t decode_workspace_bytes(const Layer& L, int B) {
  const int na = B * L.k + B;
  size_t z = al(sizeof(float) * B * L.E) + al(sizeof(int)) +
             al(sizeof(int) * (L.E + 1)) + al(sizeof(int) * (L.E + 2)) + al(sizeof(int) * na) +
             al(sizeof(float) * na) + al(sizeof(float) * B * (L.k + 1) * L.f);
  if (L.prec == MOE_MXFP8)
    z += al(2 * (size_t)B * L.d) + al((size_t)B * L.d / 32) + al(2 * (size_t)B * (L.k + 1) * L.f) +
         al((size_t)B * (L.k + 1) * L.f / 32);
  return z;
}

cudaError_t launch_decode_route(const Layer& L, const void* x, int B, void* ws, cudaStream_t s) {
  DecodeWs w = carve(L, B, ws);
  // warps per logit: enough for about eight warps per SM, at most one block's eight
  int parts = 1;
  while (parts < kRouteWarps && (long)B * L.E * parts * 2 <= (long)L.num_sms * kRouteWarps) parts *= 2;
  const int items_per_block = kRouteWarps / parts;
  const int route_blocks = (B * L.E + items_per_block - 1) / items_per_block;
  decode_logits_kernel<<<route_blocks, kRouteWarps * 32, 0, s>>>((const bf16*)x, (const bf16*)L.Wr, B, L.d, L.E,
                                                                 parts, w, L.prec == MOE_MXFP8 ? 1 : 0);
  MOE_TRY(cudaGetLastError());
  return launch_pdl(decode_select_kernel, 1, kRouteWarps * 32, 0, s, L.bias, B, L.E, L.k, L.S, L.router, L.renorm,
                    L.scale, w);
}

cudaError_t launch_decode_gateup(const Layer& L, const void* x, int B, void* ws, cudaStream_t s) {
  DecodeWs w = carve(L, B, ws);
  if (B == 1)   // one token per expert
    return launch_pdl(decode_gateup_kernel<1, 10>, L.num_sms * 4, 256, 0, s, (const bf16*)x, (const bf16*)L.W13, L.d,
                      L.f, L.G, L.k, L.E, L.S, w);
  return launch_pdl(decode_gateup_kernel<kTokGroup, kBatch>, L.num_sms * 4, 256, 0, s, (const bf16*)x,
                    (const bf16*)L.W13, L.d, L.f, L.G, L.k, L.E, L.S, w);
}

cudaError_t launch_decode_gateup_mx(const Layer& L, int B, void* ws, cudaStream_t s) {
  DecodeWs w = carve(L, B, ws);
  // one token per pass over a row (an expert with several tokens re-reads its rows, from L2): the
  // registers go to a deeper load batch, faster at every B measured (1-64)
  return launch_pdl(decode_gateup_mx_kernel<1, 7>, L.num_sms * 4, 256, 0, s, (const uint8_t*)L.W13q,
                    (const uint8_t*)L.W13s, L.d, L.f, L.G, L.k, L.E, L.S, w);
}

cudaError_t launch_decode_quant_h_mx(const Layer& L, int B, void* ws, cudaStream_t s) {
  DecodeWs w = carve(L, B, ws);
  const int nblocks = B * (L.k + 1) * L.f / 32;
  return launch_pdl(decode_quant_h_kernel, (nblocks + 255) / 256, 256, 0, s, nblocks, w);
}

// Shared memory of the MXFP8 down kernel that stages h, in bytes.
size_t down_mx_stage_bytes(const Layer& L, int B) {
  constexpr int NC = 3;
  const size_t na = (size_t)B * (L.k + 1);
  return (((size_t)kDownWarps * B * NC + 3) & ~(size_t)3) * sizeof(float) + na * L.f * 2 + na * (L.f / 32);
}

bool decode_down_mx_stages_h(const Layer& L, int B) { return down_mx_stage_bytes(L, B) <= 112 * 1024; }

cudaError_t launch_decode_down_mx(const Layer& L, int B, void* y, void* ws, cudaStream_t s) {
  DecodeWs w = carve(L, B, ws);
  // three columns per warp: the d / 24 blocks fit one wave at two blocks per SM
  constexpr int NC = 3;
  const int blocks = (L.d + kDownWarps * NC - 1) / (kDownWarps * NC);
  if (decode_down_mx_stages_h(L, B)) {
    static bool attr = false;
    if (!attr) {
      MOE_TRY(cudaFuncSetAttribute(decode_down_mx_kernel<NC, 2, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   112 * 1024));
      attr = true;
    }
    return launch_pdl(decode_down_mx_kernel<NC, 2, true>, blocks, kDownWarps * 32, down_mx_stage_bytes(L, B), s,
                      (const uint8_t*)L.Wdq, (const uint8_t*)L.Wds, B, L.d, L.f, L.k, w, (bf16*)y);
  }
  return launch_pdl(decode_down_mx_kernel<NC, 2, false>, blocks, kDownWarps * 32, sizeof(float) * kDownWarps * B * NC,
                    s, (const uint8_t*)L.Wdq, (const uint8_t*)L.Wds, B, L.d, L.f, L.k, w, (bf16*)y);
}

cudaError_t launch_decode_down(const Layer& L, int B, void* y, void* ws, cudaStream_t s) {
  DecodeWs w = carve(L, B, ws);
  const int down_blocks = (L.d + kDownWarps * kCols - 1) / (kDownWarps * kCols);
  const size_t smem = sizeof(float) * kDownWarps * B * kCols;
  return launch_pdl(decode_down_kernel, down_blocks, kDownWarps * 32, smem, s, (const bf16*)L.Wd, B, L.d, L.f, L.k, w,
                    (bf16*)y);
}

}  // namespace moe
