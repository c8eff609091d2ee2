// The opaque handle behind moe_handle (internal to the library).
#pragma once
#include <vector>

#include "kernels.h"

struct ProfRec {
  int group, kernels;
  cudaEvent_t a, b;
};

struct moe_handle_s {
  moe_config cfg;
  moe::Layer L;
  int device;
  bool tc;         // bf16 tensor-core path available for this shape
  bool mx;         // MXFP8 tensor-core path (cfg.prec == MOE_MXFP8)
  bool tc_router;  // router logits on the tensor cores
  bool prof = false;
  long long launches = 0;
  std::vector<ProfRec> recs;
  std::vector<cudaEvent_t> pool;
  // Side stream: the router backward and the dx gather-sum run beside the dx and weight-gradient
  // GEMMs, and in a chunked step the next chunk's routing beside this chunk's expert GEMMs (fork /
  // join with these events; capturable in a CUDA graph).
  // moe_decode runs the grouped-GEMM forward for B >= decode_gemm_from (the measured crossover)
  int decode_gemm_from = moe::kDecodeGemmFrom;   // (MXFP8 layers: kDecodeGemmFromMx)
  cudaStream_t side = nullptr;
  cudaEvent_t ev_dh = nullptr, ev_dx = nullptr, ev_join = nullptr;
};

// api.cu: the routing steps of moe_route (router logits, top-k, counts, offsets, permutation) into
// the arrays of B, with the router GEMM's split-K partials in part (part_bytes); the no-allocation
// entry point runs exactly these steps.
moe_status route_steps(moe_handle_s* h, const moe::Bufs& B, const void* x, float* part, size_t part_bytes,
                       cudaStream_t s);
