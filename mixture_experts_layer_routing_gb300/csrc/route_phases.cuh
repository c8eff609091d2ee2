// Counts, offsets and the stable dispatch permutation as block-level device
// functions: the routing kernels of route.cu run them one block per chunk (or
// one block for the scan), and the whole-forward persistent kernel runs the
// same functions as phases between its grid-wide barriers, so both produce the
// same integers.
//
// Assignments a = t*k + j are cut into chunks of kChunk. (1) each chunk counts
// its experts; (2) one block turns the chunk counts into expert counts, the
// exclusive offsets, per-chunk bases and the tile prefixes; (3) each chunk
// ranks its assignments stably (warp match + per-warp counts, in passes of the
// block's size) and writes the permutation. Integer-only and
// order-independent: bit-exact every run. Follows "Cursor открыл код ядра
// Mixture of Experts ..." (dzen.guru), section "Три решения, которые дали
// результат": the CPU is out of the loop and sizes no buffer; nothing is
// dropped.
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace moe {

// Shared-memory words each function needs (ints).
constexpr int kHistSmem = kMaxE;
constexpr int kScanSmem = (kMaxE + 1) + 16 * 7 + 4;
__host__ __device__ constexpr int permute_smem(int nwarps) { return nwarps * kMaxE + kMaxE; }

// Chunk ch: chunk_hist[ch][e] = number of its assignments routed to e. Any block size.
__device__ __forceinline__ void hist_chunk(const int* __restrict__ idx, int A, int E, int ch,
                                           int* __restrict__ chunk_hist, int* status, int* h) {
  for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
  __syncthreads();
  const int a0 = ch * kChunk;
  for (int a = a0 + threadIdx.x; a < min(A, a0 + kChunk); a += blockDim.x) {
    const int e = idx[a];
    if ((unsigned)e >= (unsigned)E) {
      set_error(status, MOE_ERR_DEVICE_INDEX);
      continue;
    }
    atomicAdd(&h[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_hist[(size_t)ch * E + e] = h[e];
  __syncthreads();
}

// One block of at least E + S threads (and at most 512). Segments 0..E-1 are the routed experts,
// segment E (when S = 1) is the shared expert with all T tokens. Writes cnt, off, the tile
// prefixes (mt_off and the kPrefixArrays - 1 arrays after it) and chunk_base.
__device__ __forceinline__ void scan_segments(const int* __restrict__ chunk_hist, int nch, int E, int S, int T,
                                              int* __restrict__ chunk_base, int* __restrict__ cnt,
                                              int* __restrict__ off, int* __restrict__ mt_off, int* sm) {
  int* c_s = sm;                                            // [kMaxE + 1]
  int (*warp_tot)[7] = reinterpret_cast<int (*)[7]>(sm + kMaxE + 1);   // [16][7]
  int* tot = sm + kMaxE + 1 + 16 * 7;                       // all tiles, candidate dense tiles, other tiles,
                                                            // other non-empty segments
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
  // exclusive scans over the block of: c, ceil(c / kBM) (tiles), ceil(tiles / 2) (pairs), the tiles
  // of dense segments and of the others, and the same split of the pairs (the GEMMs whose CTAs take
  // two 128-row tiles of a segment at once)
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
  __syncthreads();
}

// Chunk ch: sorted position of each of its assignments (ascending a within an expert), in passes of
// blockDim (a multiple of 32) assignments. sm: permute_smem(blockDim / 32) ints.
__device__ __forceinline__ void permute_chunk(const int* __restrict__ idx, const float* __restrict__ gate, int A,
                                              int E, int k, int ch, const int* __restrict__ chunk_base,
                                              int* __restrict__ perm, int* __restrict__ inv,
                                              int* __restrict__ row_token, float* __restrict__ row_gate, int* sm) {
  const int nw = blockDim.x >> 5;
  int* wcnt = sm;                 // [nw][kMaxE] per-warp count of each expert in this pass
  int* run = sm + nw * kMaxE;     // [kMaxE] assignments of each expert in earlier passes
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  for (int e = tid; e < E; e += blockDim.x) run[e] = 0;
  for (int p0 = 0; p0 < kChunk; p0 += blockDim.x) {
    for (int i = tid; i < nw * kMaxE; i += blockDim.x) wcnt[i] = 0;
    __syncthreads();
    const int a = ch * kChunk + p0 + tid;
    const bool valid = p0 + tid < kChunk && a < A;
    int e = valid ? idx[a] : -1;
    if (valid && (unsigned)e >= (unsigned)E) e = -1;   // reported by hist_chunk
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const int rank_in_warp = __popc(same & ((1u << lane) - 1u));
    if (e >= 0 && rank_in_warp == 0) wcnt[w * kMaxE + e] = __popc(same);
    __syncthreads();
    if (e >= 0) {
      int before = run[e];
      for (int q = 0; q < w; ++q) before += wcnt[q * kMaxE + e];
      const int p = chunk_base[(size_t)ch * E + e] + before + rank_in_warp;
      perm[p] = a;
      inv[a] = p;
      row_token[p] = a / k;
      row_gate[p] = gate ? gate[a] : 1.0f;
    }
    __syncthreads();
    for (int e2 = tid; e2 < E; e2 += blockDim.x) {
      int s = 0;
      for (int q = 0; q < nw; ++q) s += wcnt[q * kMaxE + e2];
      run[e2] += s;
    }
    __syncthreads();
  }
}

}  // namespace moe
