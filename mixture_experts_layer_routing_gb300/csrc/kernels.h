// Internal interface between the host API (api.cu) and the kernel translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kMaxE = 256;        // routed experts supported by the routing kernels
constexpr int kMaxK = 8;          // experts per token
constexpr int kChunk = 1024;      // assignments per block of the histogram / permutation kernels
constexpr int kBM = 128;          // rows per M-tile of the grouped GEMMs (segment padding unit)
constexpr int kRouterSplit = 8;   // most row splits of an expert segment in the router weight gradient
constexpr int kRouterSplitRows = 256;   // rows per split
// Segments with kDenseTiles M-tiles or more reuse each weight byte for >= 384 rows, above the
// bf16 ridge of about 280 flop/byte: candidates for the "dense" tile stream (see scan_kernel).
constexpr int kDenseTiles = 3;
constexpr int kPrefixArrays = 6;   // tile-schedule prefix arrays of nseg + 1 ints each (Bufs::mt_off)
constexpr int kGate = 128;        // gate/up interleave block of the packed bf16 W13 (rows)
constexpr int kGateMx = 64;       // gate/up interleave block of the MXFP8 W13 (rows)
constexpr int kMaxDecodeB = 64;
constexpr int kDecodeGemmFrom = 4;     // batch size from which moe_decode takes the grouped-GEMM forward (bf16)
constexpr int kDecodeGemmFromMx = 4;   // (MXFP8)

// Shape of one layer and the pointers that stay fixed after moe_set_weights.
struct Layer {
  int d, E, S, f, k, router, renorm, prec;
  float scale;
  int G;                 // gate/up interleave block actually used (kGate, or f when f < kGate)
  // packed weights (device)
  void* W13;             // [E+S][2f][d] gate/up rows interleaved in blocks of G
  void* Wd;              // [E+S][d][f]
  void* Wr;              // [E][d]
  float* bias;           // [E]
  int* status;           // device status word
  int num_sms;
  bool has_weights;
  // tensor maps of the packed weights (bf16 tcgen05 path)
  CUtensorMap tm_W13;       // K-major rows of W13 (box 64 x 256)
  CUtensorMap tm_Wd;        // K-major rows of Wd (box 64 x 256)
  CUtensorMap tm_W13_mn;    // W13 as [K=2f rows][N=d] for dx (box 64 x 64)
  CUtensorMap tm_Wd_mn;     // Wd as [K=d rows][N=f] for the dY.Wd product (box 64 x 64)
  CUtensorMap tm_W13_h;     // K-major rows of W13, box 64 x 128 (half an n-tile: one CTA of a pair)
  CUtensorMap tm_Wd_h;      // K-major rows of Wd, box 64 x 128
  int pairs;                // 1: expert GEMMs on 2-SM CTA pairs; 0 (default): one CTA per tile
  int fused;                // 1: forward gate/up and down GEMMs as one persistent kernel; 2: the whole forward
  int row_tiles;            // 128-row tiles per CTA of the bf16 segment GEMMs over token rows (1 or 2)
  unsigned* dep;            // fused kernels: per-m-tile arrival counters (zero between calls)
  int dep_len;              // their number
  unsigned* dep_done;       // fused kernels: [0] tile queue head, [1] CTAs finished, [2] gate/up epilogue warps
                            // finished, [3] grid-barrier arrivals, [4] abort (zero between calls)
  // MXFP8 packed weights: E4M3 codes and E8M0 scales (one per 32 along the named axis)
  // MXFP8 scales: K-major arrays row-major (rows, K/32); MN-major arrays (Krows/32, W) stored
  // as [Krows/128][W][4] (the four scales of a column's 128-row K block in one word).
  // scales in 512-byte atoms (mx_quant.cuh: atom_k for the K-major copies, atom_mn for the others)
  uint8_t *W13q, *W13s;     // [E+S][2f][d] along d (gate/up interleaved in blocks of kGateMx rows)
  uint8_t *W13c, *W13cs;    // same rows quantised along the packed 2f rows
  uint8_t *Wdq, *Wds;       // [E+S][d][f] along f
  uint8_t *Wdc, *Wdcs;      // same rows quantised along d
  CUtensorMap tm_W13q, tm_Wdq, tm_W13c, tm_Wdc;
};

// Device buffers of one forward / backward, carved from the caller's workspace and context.
struct Bufs {
  int T, A, R;           // tokens, assignments (T*k), sorted rows (A + S*T)
  int nch;               // histogram chunks
  // routing (context when training, else workspace)
  float* logits;         // [T, E]
  int* idx;              // [T, k]
  float* gate;           // [T, k]
  int* cnt;              // [E+S]
  int* off;              // [E+S+1]
  int* mt_off;           // [E+S+1] prefix of ceil(cnt / kBM), then [E+S+1] each: prefixes of
                         // pairs of tiles, of the tiles of dense segments and of the others, of
                         // the pairs of dense segments and of the others (kPrefixArrays in all)
  int* perm;             // [A]
  int* inv;              // [A]
  int* row_token;        // [R]
  float* row_gate;       // [R]
  void* uv;              // [R, 2f] saved pre-activations (interleaved like W13), may be null
  // forward scratch
  int* chunk_hist;       // [nch, E]
  int* chunk_base;       // [nch, E]
  void* h;               // [R, f]
  void* o;               // [R, d]
  // backward scratch
  void* dudv;            // [R, 2f]
  void* hg;              // [R, f]  gate * h
  float* dg_part;        // [A, f / 64] gate-gradient partials, one per 64 features
  void* dx_rows;         // [R, d]
  float* dl;             // [T, E]
  float* dwr_part;       // [kRouterSplit, E, d] router weight-gradient partials
  float* dgate;          // [T, k]
  // MXFP8 operands (codes, scales)
  // codes in expert-sorted row order, scale atoms by row tile (atom_tile, Rp rows)
  uint8_t *xq, *xs;      // [R, d]: x of each sorted row
  uint8_t *hq, *hs;      // [R, f]
  uint8_t *dyq, *dys;    // [R, d]: dy of each sorted row
  uint8_t *dudvq, *dudvs;  // [R, 2f]
  int Rp_max;            // rows of the token-axis operands: each segment padded to 128 (upper bound)
  const int* tok_k32;    // chunked step (nullable): 32-row blocks of each segment's token-axis rows, whose
                         // chunks are packed at 32 rows (the rest of its last 128-row group is unused)
  uint8_t *dudv_t, *dudv_ts, *x_t, *x_ts, *dy_t, *dy_ts, *hg_t, *hg_ts;  // [Rp, W], atom_mn scales
};

// ----------------------------------------------------------- launchers
// route.cu
cudaError_t launch_router_logits(const Layer& L, const void* x, int T, float* logits, cudaStream_t s);
cudaError_t launch_topk(const Layer& L, const float* logits, int T, int* idx, float* gate, cudaStream_t s);
cudaError_t launch_scan_permute(const Layer& L, const Bufs& B, cudaStream_t s);
// simt.cu (fp32 path and reference-grade kernels)
cudaError_t launch_simt_gateup(const Layer& L, const Bufs& B, const void* x, cudaStream_t s);
cudaError_t launch_simt_down(const Layer& L, const Bufs& B, cudaStream_t s);
cudaError_t launch_simt_bwd_dh(const Layer& L, const Bufs& B, const void* dy, cudaStream_t s);
cudaError_t launch_simt_bwd_dx(const Layer& L, const Bufs& B, cudaStream_t s);
cudaError_t launch_simt_bwd_dw13(const Layer& L, const Bufs& B, const void* x, void* dWg, void* dWu, bool acc,
                                cudaStream_t s);
cudaError_t launch_simt_bwd_dwd(const Layer& L, const Bufs& B, const void* dy, void* dWd, bool acc, cudaStream_t s);
// combine.cu
cudaError_t launch_combine(const Layer& L, const Bufs& B, void* y, cudaStream_t s);
cudaError_t launch_router_bwd(const Layer& L, const Bufs& B, const void* x, float* dWr, bool acc, cudaStream_t s);
cudaError_t launch_dx_gather(const Layer& L, const Bufs& B, void* dx, cudaStream_t s);
cudaError_t launch_pack_weights(const Layer& L, const void* Wr, const float* bias, const void* Wg,
                                const void* Wu, const void* Wd, cudaStream_t s);
// decode.cu
size_t decode_workspace_bytes(const Layer& L, int B);
cudaError_t launch_decode_route(const Layer& L, const void* x, int B, void* ws, cudaStream_t s);
cudaError_t launch_decode_gateup(const Layer& L, const void* x, int B, void* ws, cudaStream_t s);
cudaError_t launch_decode_down(const Layer& L, int B, void* y, void* ws, cudaStream_t s);
// MXFP8 layers: x quantised along d, gate/up on E4M3 W13, h quantised along f, down on E4M3 Wd.
cudaError_t launch_decode_gateup_mx(const Layer& L, int B, void* ws, cudaStream_t s);
cudaError_t launch_decode_quant_h_mx(const Layer& L, int B, void* ws, cudaStream_t s);
cudaError_t launch_decode_down_mx(const Layer& L, int B, void* y, void* ws, cudaStream_t s);
bool decode_down_mx_stages_h(const Layer& L, int B);   // the down kernel quantises h itself (no h quantiser)
// tc_gemm.cu (bf16 tcgen05 path)
bool tc_supported(const Layer& L);
cudaError_t tc_init(Layer& L);   // encodes the weight tensor maps, sets kernel attributes
// part (nullable, part_bytes): scratch for split-K partials when T gives few row tiles
constexpr size_t kRouterPartBytes = 24u << 20;   // router split-K partials, at most (2 splits of T = 12288, E = 256)
int tc_router_splits(const Layer& L, int T);
cudaError_t launch_tc_router_logits(const Layer& L, const void* x, int T, float* logits, cudaStream_t s,
                                    float* part, size_t part_bytes);
cudaError_t launch_tc_gateup(const Layer& L, const Bufs& B, const void* x, cudaStream_t s);
cudaError_t launch_tc_down(const Layer& L, const Bufs& B, cudaStream_t s);
cudaError_t launch_tc_fused_experts(const Layer& L, const Bufs& B, const void* x, cudaStream_t s);
cudaError_t launch_tc_fused_forward(const Layer& L, const Bufs& B, const void* x, void* y, cudaStream_t s);
cudaError_t launch_tc_bwd_dh(const Layer& L, const Bufs& B, const void* dy, cudaStream_t s);
cudaError_t launch_tc_bwd_dx(const Layer& L, const Bufs& B, cudaStream_t s);
cudaError_t launch_tc_bwd_dw13(const Layer& L, const Bufs& B, const void* x, void* dWg, void* dWu, bool acc,
                              cudaStream_t s);
cudaError_t launch_tc_bwd_dwd(const Layer& L, const Bufs& B, const void* dy, void* dWd, bool acc, cudaStream_t s);

// mx.cu (MXFP8 tcgen05 path)
bool mx_supported(const Layer& L);
size_t mx_packed_bytes(const Layer& L);
cudaError_t mx_pack_weights(Layer& L, const void* Wg, const void* Wu, const void* Wd, void* base, cudaStream_t s);
cudaError_t launch_mx_quant_sorted(const Layer& L, const Bufs& B, const void* src, int K, uint8_t* q, uint8_t* s,
                                   cudaStream_t st);
cudaError_t launch_mx_quant_tokens(const Layer& L, const Bufs& B, const void* src, int W, uint8_t* q, uint8_t* s,
                                   cudaStream_t st, const int* out_base = nullptr);
cudaError_t launch_mx_chunk_layout(const Layer& L, const int* chunk_off, int n, int* comb_base, int* comb_mt,
                                   int* comb_k32, cudaStream_t st);
cudaError_t launch_mx_gateup(const Layer& L, const Bufs& B, cudaStream_t s);
cudaError_t launch_mx_down(const Layer& L, const Bufs& B, cudaStream_t s);
// dY.Wd with the SwiGLU backward: du/dv quantised along 2f into B (dx's operand) and, with g * h,
// along the token axis into O's token-axis buffers (rows from tok_base[e], or mt_off[e] * 128 when null)
cudaError_t launch_mx_bwd_dh(const Layer& L, const Bufs& B, const Bufs& O, const int* tok_base, cudaStream_t s);
cudaError_t launch_mx_bwd_dx(const Layer& L, const Bufs& B, cudaStream_t s);
cudaError_t launch_mx_bwd_dw13(const Layer& L, const Bufs& B, void* dWg, void* dWu, bool acc, cudaStream_t s);
cudaError_t launch_mx_bwd_dwd(const Layer& L, const Bufs& B, void* dWd, bool acc, cudaStream_t s);
bool tc_router_supported(const Layer& L);

// Storage bytes of activations, outputs and bf16 weights (MXFP8 layers take bf16 activations).
inline size_t elem_bytes(int prec) { return prec == MOE_FP32 ? 4 : 2; }

}  // namespace moe
