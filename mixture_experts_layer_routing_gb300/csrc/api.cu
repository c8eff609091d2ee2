// Host side of the C ABI declared in include/moe.h: validation, workspace
// carving and the launch sequence of each call. Every call only enqueues work
// on the caller's stream; nothing here waits for the device except
// moe_get_status.
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include "common.cuh"
#include "handle.h"
#include "kernels.h"

using namespace moe;

// Kernel groups reported by moe_profile_read.
enum Group {
  G_ROUTER_LOGITS, G_TOPK, G_SCAN_PERMUTE, G_GATEUP, G_DOWN, G_COMBINE, G_BWD_DH, G_BWD_DX, G_ROUTER_BWD,
  G_DX_GATHER, G_BWD_DW13, G_BWD_DWD, G_DECODE_ROUTE, G_DECODE_GATEUP, G_DECODE_DOWN, G_PACK, G_MX_QUANT, G_FUSED, G_COUNT
};
static const char* kGroupNames[G_COUNT] = {
    "router_logits", "topk", "scan_permute", "gateup", "down", "combine", "bwd_dh", "bwd_dx", "router_bwd",
    "dx_gather", "bwd_dw13", "bwd_dwd", "decode_route", "decode_gateup", "decode_down", "pack_weights", "mx_quant",
    "experts_fused"};

namespace {

inline size_t al(size_t v) { return (v + 255) & ~size_t(255); }

// Rows of the token-axis MXFP8 operands: every segment padded to 128 rows (upper bound over routings).
size_t rp_max(const Layer& L, int T) {
  const size_t R = (size_t)T * L.k + (size_t)L.S * T;
  return (R + 127) / 128 * 128 + 128 * (size_t)(L.E + L.S);
}

struct Sizes {
  size_t route, uv, fwd_scratch, ctx, fwd_ws, bwd_ws, packed;
};

Sizes sizes_for(const Layer& L, int T) {
  const size_t A = (size_t)T * L.k, nseg = L.E + L.S, R = A + (size_t)L.S * T;
  const size_t eb = elem_bytes(L.prec);
  const size_t nch = (A + kChunk - 1) / kChunk;
  Sizes z;
  z.route = al(4 * T * (size_t)L.E) + 2 * al(4 * A) + 2 * al(4 * (nseg + 1)) + al(4 * kPrefixArrays * (nseg + 1)) + 2 * al(4 * A) +
            2 * al(4 * R);
  z.uv = al(eb * R * 2 * L.f);
  z.fwd_scratch = 2 * al(4 * nch * L.E) + al(eb * R * L.f) + al(eb * R * L.d);
  z.ctx = z.route + z.uv;
  z.fwd_ws = z.route + z.fwd_scratch;
  z.bwd_ws = al(eb * R * 2 * L.f) + al(eb * R * L.f) + al(4 * A * (L.f / 64)) + al(eb * R * L.d) +
             al(4 * T * (size_t)L.E) + al(4 * A) + al(4 * (size_t)kRouterSplit * L.E * L.d);
  if (L.prec == MOE_MXFP8) z.bwd_ws -= al(eb * R * 2 * L.f) + al(eb * R * L.f);   // no bf16 du/dv, g * h
  z.packed = al(eb * nseg * 2 * L.f * L.d) + al(eb * nseg * L.d * L.f) + al(eb * L.E * L.d) + al(4 * L.E);
  if (L.prec == MOE_MXFP8) {
    const size_t d = L.d, f = L.f, Rp = rp_max(L, T);
    // activations: codes in expert-sorted row order [R], scale atoms per 128-row tile (Rp rows)
    z.fwd_scratch = 2 * al(4 * nch * L.E) + al(R * d) + al(Rp * d / 32) + al(R * f) + al(Rp * f / 32) + al(2 * R * d);
    z.fwd_ws = z.route + z.fwd_scratch;
    z.bwd_ws += al(R * d) + al(Rp * d / 32) + al(R * 2 * f) + al(Rp * 2 * f / 32) + al(Rp * 2 * f) +
                al(Rp * 2 * f / 32) + 2 * (al(Rp * d) + al(Rp * d / 32)) + al(Rp * f) + al(Rp * f / 32);
    z.packed = mx_packed_bytes(L) + al(2 * L.E * d) + al(4 * L.E);
  }
  if (L.prec != MOE_FP32) {   // decode uses the forward workspace
    const size_t dec = decode_workspace_bytes(L, T < kMaxDecodeB ? T : kMaxDecodeB);
    if (dec > z.fwd_ws) z.fwd_ws = dec;
  }
  return z;
}

// Routing arrays at p (in context or workspace order); returns the end.
char* carve_route(Bufs& B, const Layer& L, char* p) {
  const size_t nseg = L.E + L.S;
  B.logits = (float*)p; p += al(4 * (size_t)B.T * L.E);
  B.idx = (int*)p; p += al(4 * (size_t)B.A);
  B.gate = (float*)p; p += al(4 * (size_t)B.A);
  B.cnt = (int*)p; p += al(4 * (nseg + 1));
  B.off = (int*)p; p += al(4 * (nseg + 1));
  B.mt_off = (int*)p; p += al(4 * kPrefixArrays * (nseg + 1));   // mt_off, then the other tile prefixes
  B.perm = (int*)p; p += al(4 * (size_t)B.A);
  B.inv = (int*)p; p += al(4 * (size_t)B.A);
  B.row_token = (int*)p; p += al(4 * (size_t)B.R);
  B.row_gate = (float*)p; p += al(4 * (size_t)B.R);
  return p;
}

Bufs carve(const Layer& L, int T, void* ws, const void* ctx, void* bws) {
  Bufs B;
  std::memset(&B, 0, sizeof(B));
  B.T = T;
  B.A = T * L.k;
  B.R = B.A + L.S * T;
  B.nch = (B.A + kChunk - 1) / kChunk;
  const size_t eb = elem_bytes(L.prec);
  char* w = (char*)ws;
  if (ctx) {
    char* c = carve_route(B, L, (char*)ctx);
    B.uv = c;
  } else if (w) {
    w = carve_route(B, L, w);
  }
  const bool mx = L.prec == MOE_MXFP8;
  const size_t d = L.d, f = L.f, R = B.R;
  if (w) {
    B.chunk_hist = (int*)w; w += al(4 * (size_t)B.nch * L.E);
    B.chunk_base = (int*)w; w += al(4 * (size_t)B.nch * L.E);
    if (mx) {
      const size_t Rp = rp_max(L, T);
      B.xq = (uint8_t*)w; w += al(R * d);
      B.xs = (uint8_t*)w; w += al(Rp * d / 32);
      B.hq = (uint8_t*)w; w += al(R * f);
      B.hs = (uint8_t*)w; w += al(Rp * f / 32);
    } else {
      B.h = w; w += al(eb * B.R * L.f);
    }
    B.o = w; w += al(eb * B.R * L.d);
  }
  if (bws) {
    char* b = (char*)bws;
    if (!mx) {   // (MXFP8 quantises du/dv and g * h in the dY.Wd epilogue)
      B.dudv = b; b += al(eb * B.R * 2 * L.f);
      B.hg = b; b += al(eb * B.R * L.f);
    }
    B.dg_part = (float*)b; b += al(4 * (size_t)B.A * (L.f / 64));
    B.dx_rows = b; b += al(eb * B.R * L.d);
    B.dl = (float*)b; b += al(4 * (size_t)B.T * L.E);
    B.dgate = (float*)b; b += al(4 * (size_t)B.A);
    B.dwr_part = (float*)b; b += al(4 * (size_t)kRouterSplit * L.E * L.d);
    if (mx) {
      const size_t Rp = rp_max(L, T);
      B.Rp_max = (int)Rp;
      B.dyq = (uint8_t*)b; b += al(R * d);
      B.dys = (uint8_t*)b; b += al(Rp * d / 32);
      B.dudvq = (uint8_t*)b; b += al(R * 2 * f);
      B.dudvs = (uint8_t*)b; b += al(Rp * 2 * f / 32);
      B.dudv_t = (uint8_t*)b; b += al(Rp * 2 * f);
      B.dudv_ts = (uint8_t*)b; b += al(Rp * 2 * f / 32);
      B.x_t = (uint8_t*)b; b += al(Rp * d);
      B.x_ts = (uint8_t*)b; b += al(Rp * d / 32);
      B.dy_t = (uint8_t*)b; b += al(Rp * d);
      B.dy_ts = (uint8_t*)b; b += al(Rp * d / 32);
      B.hg_t = (uint8_t*)b; b += al(Rp * f);
      B.hg_ts = (uint8_t*)b; b += al(Rp * f / 32);
    }
  }
  return B;
}

inline bool aligned256(const void* p) { return ((uintptr_t)p & 255) == 0; }
inline bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

#define CK(expr)                                  \
  do {                                            \
    if ((expr) != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

cudaEvent_t take_event(moe_handle_s* h) {
  if (!h->pool.empty()) {
    cudaEvent_t e = h->pool.back();
    h->pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Launches one kernel group (nk kernels) and, when profiling, brackets it with events on s.
template <class F>
cudaError_t run(moe_handle_s* h, cudaStream_t s, int group, int nk, F&& f) {
  cudaEvent_t a = nullptr, b = nullptr;
  if (h->prof) {
    a = take_event(h);
    b = take_event(h);
    if (a && b) cudaEventRecord(a, s);
  }
  const cudaError_t e = f();
  if (a && b) {
    cudaEventRecord(b, s);
    h->recs.push_back({group, nk, a, b});
  }
  h->launches += nk;
  return e;
}

void destroy_side(moe_handle_s* h) {
  if (h->ev_dh) cudaEventDestroy(h->ev_dh);
  if (h->ev_dx) cudaEventDestroy(h->ev_dx);
  if (h->ev_join) cudaEventDestroy(h->ev_join);
  if (h->side) cudaStreamDestroy(h->side);
  h->side = nullptr;
  h->ev_dh = h->ev_dx = h->ev_join = nullptr;
}

moe_status check_T(const moe_handle_s* h, int T) {
  if (T < 0 || T > h->cfg.T_max) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// router logits, top-k, counts, offsets, permutation. part (nullable): where the router GEMM's
// split-K partials go; by default the forward scratch o, which is not yet written at this point.
moe_status run_route(moe_handle_s* h, const Bufs& B, const void* x, const float* logits_override,
                     cudaStream_t s, float* part = nullptr, size_t part_bytes = 0) {
  const Layer& L = h->L;
  const float* lg = B.logits;
  if (logits_override) {
    lg = logits_override;
  } else if (h->tc_router) {
    if (!part) {
      part = (float*)B.o;
      part_bytes = B.o ? (size_t)B.R * L.d * elem_bytes(L.prec) : 0;
    }
    const int nk = tc_router_splits(L, B.T) > 1 ? 2 : 1;
    CK(run(h, s, G_ROUTER_LOGITS, nk,
           [&] { return launch_tc_router_logits(L, x, B.T, B.logits, s, part, part_bytes); }));
  } else {
    CK(run(h, s, G_ROUTER_LOGITS, 1, [&] { return launch_router_logits(L, x, B.T, B.logits, s); }));
  }
  CK(run(h, s, G_TOPK, 1, [&] { return launch_topk(L, lg, B.T, B.idx, B.gate, s); }));
  CK(run(h, s, G_SCAN_PERMUTE, L.S ? 4 : 3, [&] { return launch_scan_permute(L, B, s); }));
  if (logits_override && lg != B.logits)
    CK(cudaMemcpyAsync(B.logits, lg, sizeof(float) * (size_t)B.T * L.E, cudaMemcpyDeviceToDevice, s));
  return MOE_OK;
}

// Combined token-axis operands of a chunked MXFP8 step (see moe_train_chunked).
struct MxDefer {
  Bufs comb;        // dudv_t, x_t, dy_t, hg_t (+ scales) over all chunks; mt_off = per-expert block prefix
  const int* base;  // [nseg] row where each expert's rows of the current chunk start
};

// The expert part of a forward of T >= 1 tokens whose routing is in ctx (or the workspace).
moe_status forward_experts(moe_handle_s* h, const void* x, int T, void* y, void* ctx, void* workspace,
                           cudaStream_t s) {
  const Layer& L = h->L;
  Bufs B = carve(L, T, workspace, ctx, nullptr);
  if (h->mx) {
    CK(run(h, s, G_MX_QUANT, 1, [&] { return launch_mx_quant_sorted(L, B, x, L.d, B.xq, B.xs, s); }));
    CK(run(h, s, G_GATEUP, 1, [&] { return launch_mx_gateup(L, B, s); }));
    CK(run(h, s, G_DOWN, 1, [&] { return launch_mx_down(L, B, s); }));
  } else if (h->tc && L.fused) {
    CK(run(h, s, G_FUSED, 1, [&] { return launch_tc_fused_experts(L, B, x, s); }));
  } else if (h->tc) {
    CK(run(h, s, G_GATEUP, 1, [&] { return launch_tc_gateup(L, B, x, s); }));
    CK(run(h, s, G_DOWN, 1, [&] { return launch_tc_down(L, B, s); }));
  } else {
    CK(run(h, s, G_GATEUP, 1, [&] { return launch_simt_gateup(L, B, x, s); }));
    CK(run(h, s, G_DOWN, 1, [&] { return launch_simt_down(L, B, s); }));
  }
  CK(run(h, s, G_COMBINE, 1, [&] { return launch_combine(L, B, y, s); }));
  return MOE_OK;
}

// Forward of T >= 1 tokens (arguments already validated).
moe_status forward_body(moe_handle_s* h, const void* x, int T, void* y, void* ctx, void* workspace, cudaStream_t s) {
  const Bufs B = carve(h->L, T, workspace, ctx, nullptr);
  if (h->tc && h->L.fused == 2) {
    CK(run(h, s, G_FUSED, 1, [&] { return launch_tc_fused_forward(h->L, B, x, y, s); }));
    return MOE_OK;
  }
  const moe_status st = run_route(h, B, x, nullptr, s);
  if (st != MOE_OK) return st;
  return forward_experts(h, x, T, y, ctx, workspace, s);
}

// Backward of T >= 1 tokens with the forward's ctx (arguments already validated). acc: add the
// weight gradients to the values already in dWr, dWg, dWu, dWd instead of overwriting them.
moe_status backward_body(moe_handle_s* h, const void* x, const void* dy, int T, const void* ctx, void* dx, float* dWr,
                         void* dWg, void* dWu, void* dWd, void* workspace, cudaStream_t s, bool acc,
                         const MxDefer* defer = nullptr) {
  const Layer& L = h->L;
  Bufs B = carve(L, T, nullptr, ctx, workspace);
  // MXFP8: the token-axis operands of the weight gradients go into this call's buffers, or (chunked
  // step) into the step's combined buffers, whose single weight-gradient pass runs after the last chunk
  const Bufs& O = defer ? defer->comb : B;
  const int* base = defer ? defer->base : nullptr;
  if (h->mx) {
    CK(run(h, s, G_MX_QUANT, 1, [&] { return launch_mx_quant_sorted(L, B, dy, L.d, B.dyq, B.dys, s); }));
    CK(run(h, s, G_BWD_DH, 1, [&] { return launch_mx_bwd_dh(L, B, O, base, s); }));
    CK(run(h, s, G_BWD_DX, 1, [&] { return launch_mx_bwd_dx(L, B, s); }));
  } else if (h->tc) {
    CK(run(h, s, G_BWD_DH, 1, [&] { return launch_tc_bwd_dh(L, B, dy, s); }));
    if (h->side && !h->prof) {
      // (with per-group profiling on, everything stays on s so that each group's events bracket
      // its own kernels)
      // the router backward needs only dY.Wd's gate-gradient partials: it runs on the side stream
      // beside the dx GEMM (whose CTAs leave an SM's threads, registers and ~35 KB of shared memory
      // free); the dx gather-sum follows dx there, beside the weight-gradient GEMMs
      CK(cudaEventRecord(h->ev_dh, s));
      CK(cudaStreamWaitEvent(h->side, h->ev_dh, 0));
      const int router_kernels = (L.router == MOE_ROUTER_SOFTMAX && !L.renorm) ? 2 : 3;
      CK(run(h, h->side, G_ROUTER_BWD, router_kernels,
             [&] { return launch_router_bwd(L, B, x, dWr, acc, h->side); }));
      CK(run(h, s, G_BWD_DX, 1, [&] { return launch_tc_bwd_dx(L, B, s); }));
      CK(cudaEventRecord(h->ev_dx, s));
      CK(cudaStreamWaitEvent(h->side, h->ev_dx, 0));
      CK(run(h, h->side, G_DX_GATHER, 1, [&] { return launch_dx_gather(L, B, dx, h->side); }));
      CK(cudaEventRecord(h->ev_join, h->side));
      CK(run(h, s, G_BWD_DW13, 1, [&] { return launch_tc_bwd_dw13(L, B, x, dWg, dWu, acc, s); }));
      CK(run(h, s, G_BWD_DWD, 1, [&] { return launch_tc_bwd_dwd(L, B, dy, dWd, acc, s); }));
      CK(cudaStreamWaitEvent(s, h->ev_join, 0));
      return MOE_OK;
    }
    CK(run(h, s, G_BWD_DX, 1, [&] { return launch_tc_bwd_dx(L, B, s); }));
  } else {
    CK(run(h, s, G_BWD_DH, 1, [&] { return launch_simt_bwd_dh(L, B, dy, s); }));
    CK(run(h, s, G_BWD_DX, 1, [&] { return launch_simt_bwd_dx(L, B, s); }));
  }
  const int router_kernels = (L.router == MOE_ROUTER_SOFTMAX && !L.renorm) ? 2 : 3;
  CK(run(h, s, G_ROUTER_BWD, router_kernels, [&] { return launch_router_bwd(L, B, x, dWr, acc, s); }));
  CK(run(h, s, G_DX_GATHER, 1, [&] { return launch_dx_gather(L, B, dx, s); }));
  if (h->mx) {
    // x and dy along the token axis (du/dv and g * h came from the dY.Wd epilogue)
    CK(run(h, s, G_MX_QUANT, 2, [&] {
      cudaError_t e = launch_mx_quant_tokens(L, B, x, L.d, O.x_t, O.x_ts, s, base);
      if (e == cudaSuccess) e = launch_mx_quant_tokens(L, B, dy, L.d, O.dy_t, O.dy_ts, s, base);
      return e;
    }));
    if (!defer) {
      CK(run(h, s, G_BWD_DW13, 1, [&] { return launch_mx_bwd_dw13(L, B, dWg, dWu, acc, s); }));
      CK(run(h, s, G_BWD_DWD, 1, [&] { return launch_mx_bwd_dwd(L, B, dWd, acc, s); }));
    }
  } else if (h->tc) {
    CK(run(h, s, G_BWD_DW13, 1, [&] { return launch_tc_bwd_dw13(L, B, x, dWg, dWu, acc, s); }));
    CK(run(h, s, G_BWD_DWD, 1, [&] { return launch_tc_bwd_dwd(L, B, dy, dWd, acc, s); }));
  } else {
    CK(run(h, s, G_BWD_DW13, 1, [&] { return launch_simt_bwd_dw13(L, B, x, dWg, dWu, acc, s); }));
    CK(run(h, s, G_BWD_DWD, 1, [&] { return launch_simt_bwd_dwd(L, B, dy, dWd, acc, s); }));
  }
  return MOE_OK;
}

// Chunking of a training step over a ring of saved activations.
struct ChunkPlan {
  int chunk, n;
  size_t slot, fwd_ws, bwd_ws, comb;   // comb: MXFP8 combined weight-gradient operands (0 otherwise)
  size_t rc;                           // rows of the combined operands
  size_t part;                         // router split-K partials of the side-stream routing (0: none)
};
ChunkPlan chunk_plan(const moe_handle_s* h, int T) {
  ChunkPlan c;
  const Layer& L = h->L;
  c.chunk = (h->cfg.chunk_tokens > 0 && h->cfg.chunk_tokens < T) ? h->cfg.chunk_tokens : T;
  c.n = c.chunk > 0 ? (T + c.chunk - 1) / c.chunk : 0;
  const Sizes z = sizes_for(L, c.chunk);
  c.slot = al(z.ctx);
  c.fwd_ws = al(z.fwd_ws);
  c.bwd_ws = al(z.bwd_ws);
  c.comb = 0;
  c.rc = 0;
  c.part = (h->side && c.n > 1) ? al(kRouterPartBytes) : 0;
  if (h->mx) {
    const size_t nseg = L.E + L.S, d = L.d, f = L.f;
    c.rc = ((size_t)T * L.k + (size_t)L.S * T + 127) / 128 * 128 + 128 * nseg * (size_t)c.n;
    c.comb = al(c.rc * 2 * f) + al(c.rc * 2 * f / 32) + 2 * (al(c.rc * d) + al(c.rc * d / 32)) + al(c.rc * f) +
             al(c.rc * f / 32) + al(4 * (size_t)c.n * (nseg + 1)) + al(4 * (size_t)c.n * nseg) + 2 * al(4 * (nseg + 1));
  }
  return c;
}

}  // namespace

// The routing steps of moe_route (same kernels, launch counts and profiling records) with the
// router's split-K partials in a buffer the caller names: moe_route_noalloc.
moe_status route_steps(moe_handle_s* h, const Bufs& B, const void* x, float* part, size_t part_bytes,
                       cudaStream_t s) {
  return run_route(h, B, x, nullptr, s, part, part_bytes);
}

extern "C" {

const char* moe_status_string(int st) {
  switch (st) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or precision";
    case MOE_ERR_WORKSPACE: return "workspace or context too small or misaligned";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_DEVICE_INDEX: return "device index out of range";
    case MOE_ERR_NO_WEIGHTS: return "weights not set";
    default: return "unknown status";
  }
}

moe_status moe_create(const moe_config* cfg, moe_handle* out) {
  if (!cfg || !out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  const moe_config& c = *cfg;
  if (c.T_max < 1 || c.d < 1 || c.E < 1 || c.f < 1 || c.k < 1 || c.k > c.E || c.k > kMaxK ||
      (c.n_shared != 0 && c.n_shared != 1) || (c.router != MOE_ROUTER_SOFTMAX && c.router != MOE_ROUTER_SIGMOID) ||
      (c.prec != MOE_FP32 && c.prec != MOE_BF16 && c.prec != MOE_MXFP8) || !std::isfinite(c.route_scale) ||
      c.route_scale <= 0.f || c.chunk_tokens < 0)
    return MOE_ERR_INVALID_ARG;
  if (c.E > kMaxE || c.f % 64 != 0 || c.d % 8 != 0 || (c.prec == MOE_MXFP8 && (c.d % 128 || c.f % 128)) ||
      (long)c.T_max * c.k >= (1L << 30))
    return MOE_ERR_UNSUPPORTED;
  moe_handle_s* h = new (std::nothrow) moe_handle_s();
  if (!h) return MOE_ERR_INVALID_ARG;
  h->cfg = c;
  h->decode_gemm_from = c.prec == MOE_MXFP8 ? kDecodeGemmFromMx : kDecodeGemmFrom;
  Layer& L = h->L;
  L.d = c.d; L.E = c.E; L.S = c.n_shared; L.f = c.f; L.k = c.k;
  L.router = c.router; L.renorm = c.renorm ? 1 : 0; L.prec = c.prec; L.scale = c.route_scale;
  L.G = (c.f % kGate == 0) ? kGate : 64;
  L.pairs = 0;
  L.fused = 0;
  L.row_tiles = 1;
  L.has_weights = false;
  if (cudaGetDevice(&h->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&L.num_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
    delete h;
    return MOE_ERR_CUDA;
  }
  // status word, decode counter, and the fused kernels' counters (8 + one per m-tile)
  const size_t max_mtiles = ((size_t)c.T_max * (c.k + c.n_shared) + 127) / 128 + c.E + c.n_shared;
  const size_t word_bytes = 256 + 4 * (8 + max_mtiles);
  int* words = nullptr;
  if (cudaMalloc(&words, word_bytes) != cudaSuccess || cudaMemset(words, 0, word_bytes) != cudaSuccess) {
    if (words) cudaFree(words);
    delete h;
    return MOE_ERR_CUDA;
  }
  L.status = words;
  L.dep_done = (unsigned*)(words + 64);   // 8 words: see Layer::dep_done
  L.dep = (unsigned*)(words + 72);
  L.dep_len = (int)max_mtiles;
  if (c.prec == MOE_MXFP8) L.G = kGateMx;
  h->tc = (c.prec == MOE_BF16) && tc_supported(L);
  h->mx = (c.prec == MOE_MXFP8) && mx_supported(L);
  if (h->tc || h->mx) {
    int lo = 0, hi = 0;
    if (cudaDeviceGetStreamPriorityRange(&lo, &hi) != cudaSuccess ||
        cudaStreamCreateWithPriority(&h->side, cudaStreamNonBlocking, hi) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_dh, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_dx, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming) != cudaSuccess) {
      destroy_side(h);
      cudaFree(words);
      delete h;
      return MOE_ERR_CUDA;
    }
  }
  h->tc_router = h->tc || h->mx;
  if (c.prec == MOE_MXFP8 && !h->mx) {
    destroy_side(h);
    cudaFree(words);
    delete h;
    *out = nullptr;
    return MOE_ERR_UNSUPPORTED;
  }
  *out = h;
  return MOE_OK;
}

moe_status moe_destroy(moe_handle h) {
  if (!h) return MOE_ERR_INVALID_ARG;
  for (auto& r : h->recs) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (auto e : h->pool) cudaEventDestroy(e);
  destroy_side(h);
  cudaFree(h->L.status);
  delete h;
  return MOE_OK;
}

moe_status moe_workspace_size(moe_handle h, int T, size_t* fwd_ws, size_t* ctx, size_t* bwd_ws, size_t* packed) {
  if (!h || T < 0) return MOE_ERR_INVALID_ARG;
  const Sizes z = sizes_for(h->L, T);
  if (fwd_ws) *fwd_ws = z.fwd_ws;
  if (ctx) *ctx = z.ctx;
  if (bwd_ws) *bwd_ws = z.bwd_ws;
  if (packed) *packed = z.packed;
  return MOE_OK;
}

moe_status moe_set_weights(moe_handle h, const void* Wr, const float* bias, const void* Wg, const void* Wu,
                           const void* Wd, void* packed, void* stream) {
  if (!h || !Wr || !Wg || !Wu || !Wd || !packed) return MOE_ERR_INVALID_ARG;
  if (!aligned256(packed)) return MOE_ERR_WORKSPACE;
  if (!aligned16(Wr) || !aligned16(Wg) || !aligned16(Wu) || !aligned16(Wd)) return MOE_ERR_INVALID_ARG;
  Layer& L = h->L;
  cudaStream_t s = (cudaStream_t)stream;
  if (h->mx) {
    // MXFP8: quantised weight copies, then the bf16 router weight and the bias
    L.W13 = L.Wd = nullptr;
    L.Wr = (char*)packed + mx_packed_bytes(L);
    L.bias = (float*)((char*)L.Wr + al(2 * (size_t)L.E * L.d));
    CK(run(h, s, G_PACK, 4, [&] { return mx_pack_weights(L, Wg, Wu, Wd, packed, s); }));
    CK(cudaMemcpyAsync(L.Wr, Wr, 2 * (size_t)L.E * L.d, cudaMemcpyDeviceToDevice, s));
    if (bias) CK(cudaMemcpyAsync(L.bias, bias, 4 * (size_t)L.E, cudaMemcpyDeviceToDevice, s));
    else CK(cudaMemsetAsync(L.bias, 0, 4 * (size_t)L.E, s));
    L.has_weights = true;
    return MOE_OK;
  }
  const size_t eb = elem_bytes(L.prec);
  const size_t nseg = L.E + L.S;
  char* p = (char*)packed;
  L.W13 = p; p += al(eb * nseg * 2 * L.f * L.d);
  L.Wd = p; p += al(eb * nseg * L.d * L.f);
  L.Wr = p; p += al(eb * L.E * L.d);
  L.bias = (float*)p;
  CK(run(h, s, G_PACK, 1, [&] { return launch_pack_weights(L, Wr, bias, Wg, Wu, Wd, s); }));
  if (h->tc) CK(tc_init(L));
  L.has_weights = true;
  return MOE_OK;
}

moe_status moe_route(moe_handle h, const void* x, int T, const float* logits_override, float* logits, int32_t* idx,
                     float* gate, int32_t* cnt, int32_t* off, int32_t* perm, int32_t* inv, void* workspace,
                     void* stream) {
  if (!h || !workspace) return MOE_ERR_INVALID_ARG;
  if (check_T(h, T) != MOE_OK) return MOE_ERR_INVALID_ARG;
  if (!logits_override && (!x || !logits)) return MOE_ERR_INVALID_ARG;
  if (!h->L.has_weights) return MOE_ERR_NO_WEIGHTS;
  if (!aligned256(workspace)) return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  const Layer& L = h->L;
  cudaStream_t s = (cudaStream_t)stream;
  Bufs B = carve(L, T, workspace, nullptr, nullptr);
  moe_status st = run_route(h, B, x, logits_override, s);
  if (st != MOE_OK) return st;
  const size_t A = (size_t)T * L.k;
  if (logits) CK(cudaMemcpyAsync(logits, B.logits, 4 * (size_t)T * L.E, cudaMemcpyDeviceToDevice, s));
  if (idx) CK(cudaMemcpyAsync(idx, B.idx, 4 * A, cudaMemcpyDeviceToDevice, s));
  if (gate) CK(cudaMemcpyAsync(gate, B.gate, 4 * A, cudaMemcpyDeviceToDevice, s));
  if (cnt) CK(cudaMemcpyAsync(cnt, B.cnt, 4 * (size_t)L.E, cudaMemcpyDeviceToDevice, s));
  if (off) CK(cudaMemcpyAsync(off, B.off, 4 * (size_t)(L.E + 1), cudaMemcpyDeviceToDevice, s));
  if (perm) CK(cudaMemcpyAsync(perm, B.perm, 4 * A, cudaMemcpyDeviceToDevice, s));
  if (inv) CK(cudaMemcpyAsync(inv, B.inv, 4 * A, cudaMemcpyDeviceToDevice, s));
  return MOE_OK;
}

moe_status moe_forward(moe_handle h, const void* x, int T, void* y, void* ctx, void* workspace, void* stream) {
  if (!h || !x || !y || !workspace) return MOE_ERR_INVALID_ARG;
  if (check_T(h, T) != MOE_OK) return MOE_ERR_INVALID_ARG;
  if (!h->L.has_weights) return MOE_ERR_NO_WEIGHTS;
  if (!aligned256(workspace) || (ctx && !aligned256(ctx))) return MOE_ERR_WORKSPACE;
  if (!aligned16(x) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  return forward_body(h, x, T, y, ctx, workspace, (cudaStream_t)stream);
}

moe_status moe_backward(moe_handle h, const void* x, const void* dy, int T, const void* ctx, void* dx, float* dWr,
                        void* dWg, void* dWu, void* dWd, void* workspace, void* stream) {
  if (!h || !x || !dy || !ctx || !dx || !dWr || !dWg || !dWu || !dWd || !workspace) return MOE_ERR_INVALID_ARG;
  if (check_T(h, T) != MOE_OK) return MOE_ERR_INVALID_ARG;
  if (!h->L.has_weights) return MOE_ERR_NO_WEIGHTS;
  if (!aligned256(workspace) || !aligned256(ctx)) return MOE_ERR_WORKSPACE;
  if (!aligned16(x) || !aligned16(dy) || !aligned16(dx)) return MOE_ERR_INVALID_ARG;
  const Layer& L = h->L;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t eb = elem_bytes(L.prec);
  const size_t nseg = L.E + L.S;
  if (T == 0) {
    CK(cudaMemsetAsync(dWr, 0, 4 * (size_t)L.E * L.d, s));
    CK(cudaMemsetAsync(dWg, 0, eb * nseg * L.f * L.d, s));
    CK(cudaMemsetAsync(dWu, 0, eb * nseg * L.f * L.d, s));
    CK(cudaMemsetAsync(dWd, 0, eb * nseg * L.d * L.f, s));
    return MOE_OK;
  }
  return backward_body(h, x, dy, T, ctx, dx, dWr, dWg, dWu, dWd, workspace, s, false);
}

moe_status moe_train_chunked_sizes(moe_handle h, int T, size_t* slot_bytes, size_t* workspace_bytes,
                                   int* n_chunks) {
  if (!h || T < 1 || T > h->cfg.T_max) return MOE_ERR_INVALID_ARG;
  const ChunkPlan c = chunk_plan(h, T);
  if (slot_bytes) *slot_bytes = c.slot;
  if (workspace_bytes) *workspace_bytes = c.fwd_ws + c.bwd_ws + c.comb + c.part;
  if (n_chunks) *n_chunks = c.n;
  return MOE_OK;
}

moe_status moe_train_chunked(moe_handle h, const void* x, const void* dy, int T, void* y, void* dx, float* dWr,
                             void* dWg, void* dWu, void* dWd, void* ring, size_t ring_bytes, void* workspace,
                             int* recomputed, void* stream) {
  if (!h || !x || !dy || !y || !dx || !dWr || !dWg || !dWu || !dWd || !ring || !workspace) return MOE_ERR_INVALID_ARG;
  if (T < 1 || T > h->cfg.T_max) return MOE_ERR_INVALID_ARG;
  if (!h->L.has_weights) return MOE_ERR_NO_WEIGHTS;
  if (!aligned256(workspace) || !aligned256(ring)) return MOE_ERR_WORKSPACE;
  if (!aligned16(x) || !aligned16(dy) || !aligned16(y) || !aligned16(dx)) return MOE_ERR_INVALID_ARG;
  const ChunkPlan c = chunk_plan(h, T);
  const size_t R = ring_bytes / c.slot;
  if (R < 1) return MOE_ERR_WORKSPACE;
  const Layer& L = h->L;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t row_bytes = elem_bytes(L.prec) * (size_t)L.d;
  char* ws_f = (char*)workspace;
  char* ws_b = ws_f + c.fwd_ws;
  auto slot_of = [&](int ch) { return (char*)ring + (size_t)(ch % R) * c.slot; };
  // MXFP8: weight-gradient operands of every chunk go to combined buffers (one gradient pass at the end)
  MxDefer defer;
  int* chunk_off = nullptr;
  if (h->mx) {
    const size_t nseg = L.E + L.S, d = L.d, f = L.f, rc = c.rc;
    char* q = ws_b + c.bwd_ws;
    std::memset(&defer.comb, 0, sizeof(Bufs));
    defer.comb.dudv_t = (uint8_t*)q; q += al(rc * 2 * f);
    defer.comb.dudv_ts = (uint8_t*)q; q += al(rc * 2 * f / 32);
    defer.comb.x_t = (uint8_t*)q; q += al(rc * d);
    defer.comb.x_ts = (uint8_t*)q; q += al(rc * d / 32);
    defer.comb.dy_t = (uint8_t*)q; q += al(rc * d);
    defer.comb.dy_ts = (uint8_t*)q; q += al(rc * d / 32);
    defer.comb.hg_t = (uint8_t*)q; q += al(rc * f);
    defer.comb.hg_ts = (uint8_t*)q; q += al(rc * f / 32);
    chunk_off = (int*)q; q += al(4 * (size_t)c.n * (nseg + 1));
    int* comb_base = (int*)q; q += al(4 * (size_t)c.n * nseg);
    defer.comb.tok_k32 = (int*)q; q += al(4 * (nseg + 1));
    defer.comb.mt_off = (int*)q;
    defer.comb.Rp_max = (int)rc;
    defer.base = comb_base;
  }
  auto span = [&](int ch, int& t0, int& Tc) {
    t0 = ch * c.chunk;
    Tc = (T - t0) < c.chunk ? (T - t0) : c.chunk;
  };
  // forward: chunk ch saves its routing and pre-activations into slot ch mod R. With a side stream
  // and at least two slots, chunk ch + 1's routing (router GEMM, top-k, counts, permutation, into its
  // own slot; split-K partials in a buffer of its own) runs on the side stream while chunk ch's expert
  // GEMMs run, forked once chunk ch's routing is done (the chunk histograms are free then) and joined
  // before chunk ch + 1's expert GEMMs. One slot would be shared by both chunks' routing arrays.
  const bool overlap = c.part && !h->prof && R >= 2;
  auto route_chunk = [&](int ch, cudaStream_t st_, float* part) {
    int t0, Tc;
    span(ch, t0, Tc);
    const Bufs Bc = carve(L, Tc, ws_f, slot_of(ch), nullptr);
    return run_route(h, Bc, (const char*)x + t0 * row_bytes, nullptr, st_, part, part ? kRouterPartBytes : 0);
  };
  float* side_part = (float*)(ws_b + c.bwd_ws + c.comb);
  if (overlap) {
    const moe_status st = route_chunk(0, s, nullptr);
    if (st != MOE_OK) return st;
  }
  for (int ch = 0; ch < c.n; ++ch) {
    int t0, Tc;
    span(ch, t0, Tc);
    const bool fork = overlap && ch + 1 < c.n;
    if (fork) {
      CK(cudaEventRecord(h->ev_dh, s));
      CK(cudaStreamWaitEvent(h->side, h->ev_dh, 0));
      const moe_status st = route_chunk(ch + 1, h->side, side_part);
      if (st != MOE_OK) return st;
      CK(cudaEventRecord(h->ev_join, h->side));
    }
    const moe_status st =
        overlap ? forward_experts(h, (const char*)x + t0 * row_bytes, Tc, (char*)y + t0 * row_bytes, slot_of(ch),
                                  ws_f, s)
                : forward_body(h, (const char*)x + t0 * row_bytes, Tc, (char*)y + t0 * row_bytes, slot_of(ch),
                               ws_f, s);
    if (st != MOE_OK) return st;
    if (fork) CK(cudaStreamWaitEvent(s, h->ev_join, 0));
    if (h->mx) {
      const Bufs Bc = carve(L, Tc, nullptr, slot_of(ch), nullptr);
      CK(cudaMemcpyAsync(chunk_off + (size_t)ch * (L.E + L.S + 1), Bc.off, 4 * (size_t)(L.E + L.S + 1),
                         cudaMemcpyDeviceToDevice, s));
    }
  }
  if (h->mx)
    CK(launch_mx_chunk_layout(L, chunk_off, c.n, (int*)defer.base, defer.comb.mt_off, (int*)defer.comb.tok_k32, s));
  // backward, last chunk first: a chunk whose slot a later chunk overwrote is recomputed
  int rec = 0;
  for (int ch = c.n - 1; ch >= 0; --ch) {
    int t0, Tc;
    span(ch, t0, Tc);
    if ((size_t)ch + R < (size_t)c.n) {
      const moe_status st = forward_body(h, (const char*)x + t0 * row_bytes, Tc, (char*)y + t0 * row_bytes,
                                         slot_of(ch), ws_f, s);
      if (st != MOE_OK) return st;
      ++rec;
    }
    MxDefer dch = defer;
    dch.base = defer.base + (size_t)ch * (L.E + L.S);
    const moe_status st =
        backward_body(h, (const char*)x + t0 * row_bytes, (const char*)dy + t0 * row_bytes, Tc, slot_of(ch),
                      (char*)dx + t0 * row_bytes, dWr, dWg, dWu, dWd, ws_b, s, ch != c.n - 1,
                      h->mx ? &dch : nullptr);
    if (st != MOE_OK) return st;
  }
  if (h->mx) {
    // one weight-gradient pass over all chunks' rows (chunk order within each expert)
    Bufs Bw = carve(L, c.chunk, nullptr, slot_of(0), ws_b);
    Bw.mt_off = defer.comb.mt_off;
    Bw.Rp_max = defer.comb.Rp_max;
    Bw.dudv_t = defer.comb.dudv_t;
    Bw.dudv_ts = defer.comb.dudv_ts;
    Bw.x_t = defer.comb.x_t;
    Bw.x_ts = defer.comb.x_ts;
    Bw.dy_t = defer.comb.dy_t;
    Bw.dy_ts = defer.comb.dy_ts;
    Bw.hg_t = defer.comb.hg_t;
    Bw.hg_ts = defer.comb.hg_ts;
    Bw.tok_k32 = defer.comb.tok_k32;
    CK(run(h, s, G_BWD_DW13, 1, [&] { return launch_mx_bwd_dw13(L, Bw, dWg, dWu, false, s); }));
    CK(run(h, s, G_BWD_DWD, 1, [&] { return launch_mx_bwd_dwd(L, Bw, dWd, false, s); }));
  }
  if (recomputed) *recomputed = rec;
  return MOE_OK;
}

moe_status moe_decode(moe_handle h, const void* x, int B, void* y, void* workspace, void* stream) {
  if (!h || !x || !y || !workspace) return MOE_ERR_INVALID_ARG;
  if (B < 1 || B > kMaxDecodeB || B > h->cfg.T_max) return MOE_ERR_INVALID_ARG;
  if (h->L.prec == MOE_FP32) return MOE_ERR_UNSUPPORTED;
  if (!h->L.has_weights) return MOE_ERR_NO_WEIGHTS;
  if (!aligned256(workspace)) return MOE_ERR_WORKSPACE;
  if (!aligned16(x) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const Layer& L = h->L;
  // from the crossover batch on, the tensor-core grouped GEMMs beat the warp-per-output kernels
  // (their per-token FMA work grows with B; the GEMMs read each expert's weights once)
  if (B >= h->decode_gemm_from && (h->tc || h->mx)) return forward_body(h, x, B, y, nullptr, workspace, s);
  CK(run(h, s, G_DECODE_ROUTE, 2, [&] { return launch_decode_route(L, x, B, workspace, s); }));
  if (L.prec == MOE_MXFP8) {
    CK(run(h, s, G_DECODE_GATEUP, 1, [&] { return launch_decode_gateup_mx(L, B, workspace, s); }));
    // at small B the down kernel quantises h itself (into shared memory)
    if (!decode_down_mx_stages_h(L, B))
      CK(run(h, s, G_MX_QUANT, 1, [&] { return launch_decode_quant_h_mx(L, B, workspace, s); }));
    CK(run(h, s, G_DECODE_DOWN, 1, [&] { return launch_decode_down_mx(L, B, y, workspace, s); }));
    return MOE_OK;
  }
  CK(run(h, s, G_DECODE_GATEUP, 1, [&] { return launch_decode_gateup(L, x, B, workspace, s); }));
  CK(run(h, s, G_DECODE_DOWN, 1, [&] { return launch_decode_down(L, B, y, workspace, s); }));
  return MOE_OK;
}

moe_status moe_set_decode_crossover(moe_handle h, int b_min) {
  if (!h || b_min < 1 || b_min > kMaxDecodeB + 1) return MOE_ERR_INVALID_ARG;
  h->decode_gemm_from = b_min;
  return MOE_OK;
}

moe_status moe_profile_enable(moe_handle h, int enable) {
  if (!h) return MOE_ERR_INVALID_ARG;
  h->prof = enable != 0;
  return MOE_OK;
}

moe_status moe_profile_read(moe_handle h, int max_groups, char* names, long long* launches, double* total_ms,
                            int* n_groups) {
  if (!h || max_groups < 0 || !n_groups || (max_groups > 0 && (!names || !launches || !total_ms)))
    return MOE_ERR_INVALID_ARG;
  double ms[G_COUNT] = {};
  long long nk[G_COUNT] = {};
  bool seen[G_COUNT] = {};
  moe_status st = MOE_OK;
  for (auto& r : h->recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess)
      st = MOE_ERR_CUDA;
    ms[r.group] += t;
    nk[r.group] += r.kernels;
    seen[r.group] = true;
    h->pool.push_back(r.a);
    h->pool.push_back(r.b);
  }
  h->recs.clear();
  int n = 0;
  for (int g = 0; g < G_COUNT && n < max_groups; ++g) {
    if (!seen[g]) continue;
    std::strncpy(names + 32 * n, kGroupNames[g], 31);
    names[32 * n + 31] = 0;
    launches[n] = nk[g];
    total_ms[n] = ms[g];
    ++n;
  }
  *n_groups = n;
  return st;
}

moe_status moe_launch_count(moe_handle h, long long* launches) {
  if (!h || !launches) return MOE_ERR_INVALID_ARG;
  *launches = h->launches;
  return MOE_OK;
}

moe_status moe_set_fused(moe_handle h, int on) {
  if (!h || on < 0 || on > 2) return MOE_ERR_INVALID_ARG;
  if (on && !h->tc) return MOE_ERR_UNSUPPORTED;
  h->L.fused = on;
  return MOE_OK;
}

moe_status moe_set_pairs(moe_handle h, int mode) {
  if (!h || mode < 0 || mode > 2) return MOE_ERR_INVALID_ARG;
  h->L.pairs = mode == 1 ? 1 : 0;
  h->L.row_tiles = mode == 2 ? 2 : 1;
  return MOE_OK;
}

moe_status moe_get_status(moe_handle h, void* stream, int* device_status) {
  if (!h || !device_status) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  int v = 0;
  CK(cudaStreamSynchronize(s));
  CK(cudaMemcpy(&v, h->L.status, sizeof(int), cudaMemcpyDeviceToHost));
  CK(cudaMemset(h->L.status, 0, sizeof(int)));
  *device_status = v;
  return MOE_OK;
}

}  // extern "C"
