// Warp-level top-k expert selection and gate computation, shared by the
// batch router and the decode router.
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace moe {

// ----------------------------------------------------------------- top-k
// One warp per token. key = l + b (fp32). k rounds of a warp arg-max: the
// largest key wins, equal keys go to the lower expert index. Slot j holds the
// j-th winner. Gates from the unbiased logits.
// Called by a full warp; writes idx_out[0..k-1] and gate_out[0..k-1] (gate_out may be null).
__device__ __forceinline__ void warp_topk_gates(const float* lr, const float* __restrict__ bias, int E, int k,
                                                int router, int renorm, float scale, int* idx_out,
                                                float* gate_out) {
  constexpr int PER = kMaxE / 32;
  const int lane = threadIdx.x & 31;
  float key[PER], lg[PER];
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    const int e = lane + 32 * q;
    lg[q] = e < E ? __ldcg(lr + e) : 0.f;   // L2 read: logits may come from other blocks
    key[q] = e < E ? lg[q] + bias[e] : -INFINITY;
  }
  unsigned taken = 0;                       // bit q: expert lane + 32q already selected
  float sel_l[kMaxK];
  int sel_e[kMaxK];
  for (int j = 0; j < k; ++j) {
    float bk = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      const int e = lane + 32 * q;
      if (e < E && !(taken >> q & 1u) && (key[q] > bk || (key[q] == bk && e < be))) {
        bk = key[q];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ok > bk || (ok == bk && oe < be)) {
        bk = ok;
        be = oe;
      }
    }
    sel_e[j] = be;
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    // fetch the unbiased logit of the winner from its owner lane
    float v = 0.f;
#pragma unroll
    for (int q = 0; q < PER; ++q)
      if (q == (be >> 5)) v = lg[q];
    sel_l[j] = __shfl_sync(0xffffffffu, v, be & 31);
  }
  // gates
  float g[kMaxK];
  if (router == MOE_ROUTER_SOFTMAX) {
    if (renorm) {
      float m = sel_l[0];
      for (int j = 1; j < k; ++j) m = fmaxf(m, sel_l[j]);
      float den = 0.f;
      for (int j = 0; j < k; ++j) {
        g[j] = expf(sel_l[j] - m);
        den += g[j];
      }
      for (int j = 0; j < k; ++j) g[j] = scale * (g[j] / den);
    } else {
      float m = -INFINITY;
#pragma unroll
      for (int q = 0; q < PER; ++q)
        if (lane + 32 * q < E) m = fmaxf(m, lg[q]);
#pragma unroll
      for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float den = 0.f;
#pragma unroll
      for (int q = 0; q < PER; ++q)
        if (lane + 32 * q < E) den += expf(lg[q] - m);
      den = warp_sum(den);
      for (int j = 0; j < k; ++j) g[j] = scale * (expf(sel_l[j] - m) / den);
    }
  } else {
    float den = 0.f;
    for (int j = 0; j < k; ++j) {
      g[j] = 1.0f / (1.0f + expf(-sel_l[j]));
      den += g[j];
    }
    for (int j = 0; j < k; ++j) g[j] = renorm ? scale * (g[j] / den) : scale * g[j];
  }
  if (lane < k) {
    float gv = 0.f;
    int ev = 0;
    for (int j = 0; j < k; ++j)
      if (j == lane) {
        gv = g[j];
        ev = sel_e[j];
      }
    idx_out[lane] = ev;
    if (gate_out) gate_out[lane] = gv;
  }
}


}  // namespace moe
