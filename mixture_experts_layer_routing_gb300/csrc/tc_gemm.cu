// bf16 grouped GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// One persistent kernel template serves every GEMM of the layer: the router
// logits, both expert projections of the forward pass, and the four grouped
// products of the backward pass (fused_experts_kernel, further down, runs the
// forward's two expert GEMMs in one launch). Per CTA (one per SM):
//   warps 0-3  producers: operands pulled by token index with 16-byte cp.async
//              into the 128-byte-swizzled layout the MMA reads (the dispatch
//              never materialises a permuted copy of x or dy), or loaded by TMA
//              when their rows are contiguous. STAGES-deep smem ring.
//   warp 8     MMA issuer: tcgen05.mma kind::f16, M=128, N=BN, K=16, fp32
//              accumulators in TMEM, double buffered (2 x BN columns).
//   warps 4-7  epilogue: tcgen05.ld of the accumulator and a fused epilogue
//              (SwiGLU, gate scale, SwiGLU backward + gate gradient, stores).
// Operands are K-major (rows contiguous along K) or MN-major (rows contiguous
// along M or N, K the row index): the backward reads the weights transposed
// and reduces the weight gradients over each expert's token segment without
// any transposed copy.
// Schedules: SEG_M, tiles over the sorted rows of each expert in groups of 16
// m-tiles (every n-tile of a group before the next), so CTAs running together
// share an expert's weight and row tiles through L2, experts with many and few
// tiles interleaved when both are numerous; DENSE, one segment, optionally
// split over K; SEG_K, tiles (segment, n, m) of a per-expert weight gradient
// whose K runs over that expert's sorted rows.
//
// Pull dispatch and one fused, deterministic call per step follow "Cursor
// открыл код ядра Mixture of Experts ..." (dzen.guru), section "Три решения,
// которые дали результат". Each output element is accumulated in one CTA in
// ascending K order, so results are bit-identical between runs. Every wait on
// an mbarrier is bounded: past the limit the kernel records MOE_ERR_TIMEOUT,
// drains its copies and MMAs, frees TMEM and returns.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "route_phases.cuh"
#include "tc_ptx.cuh"
#include "topk.cuh"
#include "launch.cuh"

namespace moe {

namespace {

constexpr int BM = 128, BK = 64;
constexpr int kSmemMax = 227 * 1024;   // dynamic shared memory per CTA
constexpr int kProducerWarps = 4, kEpiWarps = 4;
constexpr int kThreads = (kProducerWarps + kEpiWarps + 1) * 32;   // 288
constexpr int kMmaWarp = kProducerWarps + kEpiWarps;               // warp 8
// Two row tiles per CTA (MT = 2): a second group of four epilogue warps (9-12) drains the second
// 128-row accumulator while warps 4-7 drain the first.
constexpr int threads_for(int MT) { return MT == 2 ? kThreads + kEpiWarps * 32 : kThreads; }   // 288 / 416

enum { A_GATHER_K = 0, A_TMA_K = 1, A_TMA_MN = 2, A_GATHER_MN = 3 };
enum { B_TMA_K = 0, B_TMA_MN = 1, B_GATHER_MN = 2 };
enum { SCHED_SEG_M = 0, SCHED_DENSE = 1, SCHED_SEG_K = 2 };
enum { EPI_SWIGLU = 0, EPI_GATE = 1, EPI_F32 = 2, EPI_DH = 3, EPI_STORE = 4, EPI_DW13 = 5, EPI_DWD = 6 };

struct TcParams {
  const bf16* A;          // gathered A rows [*, lda]     (A_GATHER_*)
  int lda;
  const bf16* Bsrc;       // gathered B rows [*, ldb]     (B_GATHER_MN)
  int ldb;
  const int* row_token;   // sorted row -> token
  const int* off;         // [nseg+1] segment row offsets
  const int* mt_off;      // [nseg+1] prefix of 128-row tiles (SEG_M)
  const int* mp_off;      // [nseg+1] prefix of pairs of 128-row tiles (SEG_M over CTA pairs)
  int nseg;               // segments scheduled (SEG_M: the first nseg segments)
  int pstride;            // entries per tile-prefix array (all segments + 1)
  int dense_rows;         // DENSE: rows of the single segment
  int K;                  // reduction length for SEG_M / DENSE (multiple of 64)
  int m_tiles;            // SEG_K: M / 128
  int n_tiles;            // N / BN
  int b_rows_per_seg;     // B by TMA: first row of segment e is e * b_rows_per_seg (SEG_M / DENSE)
  void* out;              // primary output (see the epilogues)
  int ldo;
  int n_valid;            // EPI_F32, EPI_DWD: columns to store
  void* out2;             // EPI_DH: g*h [R, f]; EPI_DW13: dWu
  const float* row_gate;  // EPI_GATE, EPI_DH
  bf16* uv;               // EPI_SWIGLU: saved pre-activations (nullable); EPI_DH: read
  int ld_uv;
  float* dg_part;         // EPI_DH: gate-gradient partials [A_rows, dg_slots]
  int dg_slots;
  int A_rows;             // routed rows (rows >= A_rows are the shared expert)
  int accumulate;         // EPI_DW13 / EPI_DWD: add to the values already in the output
  int ksplit;             // DENSE: K splits (1: none); split s writes part + s * dense_rows * ldo
  float* part;            // DENSE split-K partial outputs (EPI_F32)
  int* status;
};

__device__ __forceinline__ void unpack8_to(const bf16* p, float* f) { unpack8(*reinterpret_cast<const uint4*>(p), f); }

// ---------------------------------------------------------------- schedule
struct Tile {
  int e, m, n;
  int row0, row_end;   // SEG_M / DENSE: output rows; SEG_K: the segment's sorted rows (the K range)
  int arow0;           // first row of the A operand loaded by TMA (SEG_M: row0)
  int nkb;             // end of the K-block range (blocks of 64)
  int kb0 = 0;         // first K block (DENSE split-K; 0 otherwise)
  int ks = 0;          // K split index (DENSE split-K)
  bool two = false;    // MT = 2: the second 128-row tile (rows row0 + 128 ..) holds rows of the segment
};

template <int SCHED, int CG, int MT = 1>
__device__ __forceinline__ int total_tiles(const TcParams& p) {
  if (SCHED == SCHED_DENSE) return ((p.dense_rows + BM - 1) / BM) * p.n_tiles * p.ksplit;
  if (SCHED == SCHED_SEG_K) return p.nseg * p.m_tiles * p.n_tiles;
  return (CG == 2 || MT == 2 ? p.mp_off[p.nseg] : p.mt_off[p.nseg]) * p.n_tiles;
}

// CTA pairs: tile L is (segment, pair of m-tiles 2j and 2j+1, n); the CTA of cluster rank r takes
// m-tile 2j + r and half of the n-tile's B columns. Pairs in groups of kRasterM / 2, every n-tile
// of a group before the next group.
__device__ __forceinline__ Tile map_tile_pair(const TcParams& p, int L, int rank) {
  Tile t;
  int lo = 0, hi = p.nseg;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (p.mp_off[mid] * p.n_tiles <= L) lo = mid; else hi = mid;
  }
  constexpr int kRasterP = kRasterM / 2;
  const int Pe = p.mp_off[lo + 1] - p.mp_off[lo];
  const int local = L - p.mp_off[lo] * p.n_tiles;
  const int g = local / (kRasterP * p.n_tiles);
  const int gp = min(kRasterP, Pe - g * kRasterP);
  const int within = local - g * kRasterP * p.n_tiles;
  t.e = lo;
  t.n = within / gp;
  t.m = 2 * (g * kRasterP + within % gp) + rank;
  t.row0 = p.off[lo] + t.m * BM;
  t.row_end = p.off[lo + 1];
  t.arow0 = t.row0;
  t.nkb = p.K / BK;
  return t;
}

template <int SCHED, int CG, int MT = 1>
__device__ __forceinline__ Tile map_tile(const TcParams& p, int L, int rank) {
  if (CG == 2) return map_tile_pair(p, L, rank);
  Tile t;
  if (SCHED == SCHED_DENSE) {
    const int nk = p.K / BK;
    t.ks = L % p.ksplit;
    const int rest = L / p.ksplit;
    t.e = 0;
    t.n = rest % p.n_tiles;
    t.m = rest / p.n_tiles;
    t.row0 = t.m * BM;
    t.row_end = p.dense_rows;
    t.arow0 = t.row0;
    t.kb0 = t.ks * nk / p.ksplit;
    t.nkb = (t.ks + 1) * nk / p.ksplit;
    return t;
  }
  if (SCHED == SCHED_SEG_K) {
    const int per = p.m_tiles * p.n_tiles;
    t.e = L / per;
    const int rem = L % per;
    t.n = rem / p.m_tiles;
    t.m = rem % p.m_tiles;
    t.row0 = p.off[t.e];
    t.row_end = p.off[t.e + 1];
    t.arow0 = t.row0;
    t.nkb = (t.row_end - t.row0 + BK - 1) / BK;
    return t;
  }
  // Segments marked dense by scan_kernel (each weight tile serves several row tiles: tensor-bound)
  // and the others (each weight tile streamed for a tile or two of rows: HBM-bound) form two tile
  // streams, interleaved in proportion: tile L is dense iff floor((L+1) Nd / N) steps, so CTAs
  // running at the same time mix both kinds and keep the tensor pipe and HBM busy together.
  // scan_kernel marks none when the mix would not pay (dense under a quarter of the tiles, or the
  // others near the ridge): then the order is segment-major, which keeps each segment's weight and
  // row tiles in L2 between uses.
  // MT = 2: the units are pairs of 128-row tiles of a segment (prefixes of pairs), one per CTA.
  const int* all = MT == 2 ? p.mt_off + p.pstride : p.mt_off;
  const int* dn = p.mt_off + (MT == 2 ? 4 : 2) * p.pstride;
  const int* sp = p.mt_off + (MT == 2 ? 5 : 3) * p.pstride;
  const long N = (long)all[p.nseg] * p.n_tiles, Nd = (long)dn[p.nseg] * p.n_tiles;
  const bool mix = Nd > 0;   // scan_kernel marks dense segments only when it chose to interleave
  const long cd = mix ? (long)L * Nd / N : 0;
  const bool is_dense = mix && (long)(L + 1) * Nd / N > cd;
  const int* pre = !mix ? all : (is_dense ? dn : sp);
  const int Lc = (int)(is_dense ? cd : L - cd);   // index within the stream
  int lo = 0, hi = p.nseg;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pre[mid] * p.n_tiles <= Lc) lo = mid; else hi = mid;
  }
  const int Me = pre[lo + 1] - pre[lo];
  const int local = Lc - pre[lo] * p.n_tiles;
  // units in groups of kRasterM / MT (kRasterM 128-row tiles), every n-tile of a group before the
  // next group: CTAs running together share the group's token rows and the expert's weight tiles
  // in L2
  constexpr int RG = kRasterM / MT;
  const int g = local / (RG * p.n_tiles);
  const int gm = min(RG, Me - g * RG);
  const int within = local - g * RG * p.n_tiles;
  t.e = lo;
  t.n = within / gm;
  t.m = MT * (g * RG + within % gm);
  t.row0 = p.off[lo] + t.m * BM;
  t.row_end = p.off[lo + 1];
  t.arow0 = t.row0;
  t.nkb = p.K / BK;
  t.two = MT == 2 && t.row0 + BM < t.row_end;
  return t;
}

// Epilogue staging for TMA stores: per epilogue warp two 32-row x 64-column bf16 sub-tiles (4 KB each).
constexpr int kStageOutBytes = kEpiWarps * 2 * 32 * 128;

// Shared memory of one CTA: a ring of NS stages (A tile + this CTA's B columns: all BN, or BN/2
// when a CTA pair shares the B tile), then staging and barriers. Single CTAs keep 4 stages (deeper
// rings measured no faster and leave no L1 for the epilogue's loads); pairs take as many as fit,
// up to 8.
template <int BN, int SCHED, int CG, int MT = 1>
struct Smem {
  static constexpr int A_BYTES = MT * BM * BK * 2;
  static constexpr int B_BYTES = (BN / CG) * BK * 2;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int OUT = SCHED == SCHED_SEG_K ? kStageOutBytes : 0;
  static constexpr int FIXED = OUT + 1024 /*align*/ + 256 /*barriers*/;
  static constexpr int NS_CAP = CG == 2 ? 8 : 4;
  static constexpr int NS = (kSmemMax - FIXED) / STAGE < NS_CAP ? (kSmemMax - FIXED) / STAGE : NS_CAP;
  static constexpr int TOTAL = NS * STAGE + FIXED;
};

template <int AMODE, int BMODE>
struct Modes {
  static constexpr bool kCpAsync = AMODE == A_GATHER_K || AMODE == A_GATHER_MN || BMODE == B_GATHER_MN;
  static constexpr int kAMn = (AMODE == A_TMA_MN || AMODE == A_GATHER_MN) ? 1 : 0;
  static constexpr int kBMn = (BMODE == B_TMA_MN || BMODE == B_GATHER_MN) ? 1 : 0;
};

// Issues one stage: A and B of K block kb of tile t.
// With CTA pairs (CG = 2) this CTA loads B columns rank*BN/2 .. of the n-tile, and every TMA load
// of either CTA completes on rank 0's full barrier (lead_full), which rank 0 arms with the bytes of
// both CTAs.
// MT = 2: the A tile holds two 128-row tiles (the second at sa + BM * 128 bytes); the second is
// loaded only when it holds rows of the segment (t.two), and the MMA reads it only then.
template <int BN, int AMODE, int BMODE, int SCHED, int CG, bool kCounted = Modes<AMODE, BMODE>::kCpAsync, int MT = 1>
__device__ __forceinline__ void load_stage(const TcParams& p, const CUtensorMap* tmA, const CUtensorMap* tmB,
                                           const Tile& t, int kb, uint32_t sa, uint32_t sb, uint32_t full_bar,
                                           const bf16* const (&gsrc)[8 * MT], const uint32_t (&gbytes)[8 * MT],
                                           int ktok, int rank, uint32_t lead_full) {
  using SM = Smem<BN, SCHED, CG, MT>;
  constexpr int BNC = BN / CG;   // B columns held by this CTA
  constexpr int kHalfA = BM * BK * 2;   // bytes of one 128-row A tile
  const uint32_t tma_bytes = (AMODE == A_TMA_K || AMODE == A_TMA_MN ? (MT == 2 && !t.two ? kHalfA : SM::A_BYTES) : 0) +
                             (BMODE == B_TMA_K || BMODE == B_TMA_MN ? SM::B_BYTES : 0);
  const int ptid = threadIdx.x;
  if (ptid == 0 && tma_bytes) {
    if (rank == 0) {
      if (kCounted) mbar_expect_tx(full_bar, CG * tma_bytes);
      else mbar_arrive_expect_tx(full_bar, CG * tma_bytes);
    }
    auto load = [&](uint32_t dst, const CUtensorMap* tm, int c0, int c1) {
      if (CG == 2) tma_load_2d_pair(dst, tm, c0, c1, lead_full);
      else tma_load_2d(dst, tm, c0, c1, full_bar);
    };
    if (AMODE == A_TMA_K) {
      load(sa, tmA, kb * BK, t.arow0);
      if (MT == 2 && t.two) load(sa + kHalfA, tmA, kb * BK, t.arow0 + BM);
    }
    if (AMODE == A_TMA_MN) {
#pragma unroll
      for (int j = 0; j < BM / 64; ++j) load(sa + j * kChunkBytes, tmA, t.m * BM + j * 64, t.row0 + kb * BK);
    }
    if (BMODE == B_TMA_K) load(sb, tmB, kb * BK, t.e * p.b_rows_per_seg + t.n * BN + rank * BNC);
    if (BMODE == B_TMA_MN) {
      const int krow = (SCHED == SCHED_SEG_K ? t.row0 : t.e * p.b_rows_per_seg) + kb * BK;
#pragma unroll
      for (int j = 0; j < BNC / 64; ++j) load(sb + j * kChunkBytes, tmB, t.n * BN + rank * BNC + j * 64, krow);
    }
  }
  if (AMODE == A_GATHER_K) {
    const int warp = ptid >> 5, lane = ptid & 31;
#pragma unroll
    for (int h = 0; h < MT; ++h) {
      if (h == 1 && !t.two) break;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int r = warp * 32 + j * 4 + (lane >> 3);
        const int c = lane & 7;
        cp_async16(sa + h * kHalfA + r * 128 + ((c ^ (r & 7)) << 4), gsrc[h * 8 + j] + kb * BK, gbytes[h * 8 + j]);
      }
    }
  }
  if (AMODE == A_GATHER_MN) {
    // 128 M columns of K row 16w + rr (token ktok of lane rr) = 2 lines: two rows per instruction
    const int warp = ptid >> 5, lane = ptid & 31;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rr = 2 * i + (lane >> 4);
      const int kk = 16 * warp + rr;
      const int tok = __shfl_sync(0xffffffffu, ktok, rr);
      const bool v = t.row0 + kb * BK + kk < t.row_end;
      const int j = (lane >> 3) & 1, q = lane & 7;
      const bf16* src = p.A + (size_t)tok * p.lda + t.m * BM + j * 64 + q * 8;
      cp_async16(sa + j * kChunkBytes + kk * 128 + ((q ^ (kk & 7)) << 4), src, v ? 16u : 0u);
    }
  }
  if (BMODE == B_GATHER_MN) {
    // Warp w copies the K rows 16w..16w+15 of this block, one whole row per instruction (4 full
    // 128-byte lines), so the gather is coalesced. ktok holds, in lanes 0..15, the token of row
    // 16w + lane (loaded two blocks ahead); it is broadcast per row.
    const int warp = ptid >> 5, lane = ptid & 31;
    constexpr int LPR = BN / 64;   // 128-byte lines per row
    constexpr int RPI = 4 / LPR;   // rows per instruction
#pragma unroll
    for (int i = 0; i < 16 / RPI; ++i) {
      const int rr = RPI * i + (lane >> 3) / LPR;
      const int kk = 16 * warp + rr;
      const int tok = __shfl_sync(0xffffffffu, ktok, rr);
      const bool v = t.row0 + kb * BK + kk < t.row_end;
      const int j = (lane >> 3) % LPR, q = lane & 7;
      const bf16* src = p.Bsrc + (size_t)tok * p.ldb + t.n * BN + j * 64 + q * 8;
      cp_async16(sb + j * kChunkBytes + kk * 128 + ((q ^ (kk & 7)) << 4), src, v ? 16u : 0u);
    }
  }
}

// ---------------------------------------------------------------- epilogues
// Gate/up: u = columns 0..BN/2 of the tile, v = BN/2..BN (one 128-feature block of each);
// h = silu(u) v stored to out, and u, v to the saved pre-activations when kept.
template <int BN>
__device__ __forceinline__ void epi_swiglu(const TcParams& p, const Tile& t, uint32_t tbase, int row, bool valid) {
  bf16* hrow = (bf16*)p.out + (size_t)row * p.ldo + t.n * (BN / 2);
  bf16* uvrow = p.uv ? p.uv + (size_t)row * p.ld_uv + t.n * BN : nullptr;
#pragma unroll 1
  for (int c0 = 0; c0 < BN / 2; c0 += 32) {
    uint32_t u[32], v[32];
    tmem_ld32(tbase + c0, u);
    tmem_ld32(tbase + BN / 2 + c0, v);
    tmem_ld_wait();
    if (valid) {
      float hf[32], uf[32], vf[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        uf[i] = __uint_as_float(u[i]);
        vf[i] = __uint_as_float(v[i]);
        hf[i] = silu_f(uf[i]) * vf[i];
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) *reinterpret_cast<uint4*>(hrow + c0 + q * 8) = pack8(hf + q * 8);
      if (uvrow) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          *reinterpret_cast<uint4*>(uvrow + c0 + q * 8) = pack8(uf + q * 8);
          *reinterpret_cast<uint4*>(uvrow + BN / 2 + c0 + q * 8) = pack8(vf + q * 8);
        }
      }
    }
  }
}

// Down (kGate: scaled by the row's gate) and dx rows: the tile's BN columns stored as bf16.
template <int BN, bool kGate>
__device__ __forceinline__ void epi_scale_store(const TcParams& p, const Tile& t, uint32_t tbase, int row,
                                                bool valid) {
  const float g = (kGate && valid) ? p.row_gate[row] : 1.f;
  bf16* orow = (bf16*)p.out + (size_t)row * p.ldo + t.n * BN;
#pragma unroll 1
  for (int c0 = 0; c0 < BN; c0 += 32) {
    uint32_t a[32];
    tmem_ld32(tbase + c0, a);
    tmem_ld_wait();
    if (valid) {
      float of[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) of[i] = g * __uint_as_float(a[i]);
#pragma unroll
      for (int q = 0; q < 4; ++q) *reinterpret_cast<uint4*>(orow + c0 + q * 8) = pack8(of + q * 8);
    }
  }
}

// ------------------------------------------------------------------ kernel
// CG = 2: launched as clusters of two CTAs on two SMs. The pair computes a 256 x BN tile with
// one tcgen05.mma.cta_group::2 per K step, issued by rank 0: each CTA stages its own 128 A rows
// and half of the B columns, so each SM moves 2/3 of the shared-memory bytes of a 128 x BN tile
// per MAC and the ring is deeper. Rank 1's MMA-warp lane relays "stage s of this CTA is full" to
// rank 0's full barrier; rank 0's commits are multicast to both CTAs' empty / accumulator-full
// barriers; both epilogues report "accumulator drained" to rank 0.
// MT = 2: each CTA computes two 128-row tiles of a segment (256 x BN) with two M = 128 MMAs per
// K step that share the stage's B tile, so a stage carries twice the MMA work for 4/3 of the
// bytes; the two accumulators fill TMEM (no double buffering) and eight epilogue warps drain them.
template <int BN, int AMODE, int BMODE, int SCHED, int EPI, int CG, int MT>
__global__ void __launch_bounds__(threads_for(MT), 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmC2, TcParams p) {
  griddep_wait();    // after the predecessor grid (launch.cuh)
  griddep_launch();
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN");
  static_assert(CG == 1 || (CG == 2 && SCHED == SCHED_SEG_M && (AMODE == A_GATHER_K || AMODE == A_TMA_K) &&
                            (BMODE == B_TMA_K || BMODE == B_TMA_MN) && BN >= 128),
                "CTA pairs: segment-M schedule, K-major A, B by TMA");
  static_assert(MT == 1 || (MT == 2 && CG == 1 && SCHED == SCHED_SEG_M && (AMODE == A_GATHER_K || AMODE == A_TMA_K) &&
                            BN == 256),
                "two row tiles per CTA: segment-M schedule, K-major A, 256-column tiles");
  using MD = Modes<AMODE, BMODE>;
  using SM = Smem<BN, SCHED, CG, MT>;
  constexpr int NS = SM::NS;
  constexpr int NACC = MT == 2 ? 1 : 2;   // accumulator buffers in TMEM
  constexpr uint32_t TMEM_COLS = 2 * BN <= 128 ? 128 : (2 * BN <= 256 ? 256 : 512);
  constexpr uint32_t IDESC = idesc_bf16(BM * CG, BN, MD::kAMn, MD::kBMn);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* stage_base = smem;
  uint8_t* out_stage = smem + NS * SM::STAGE;     // SEG_K epilogue staging (1024-aligned)
  uint64_t* bars = (uint64_t*)(out_stage + SM::OUT);
  // bars: full[NS], empty[NS], tfull[2], tempty[2], drain
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + NS);
  const uint32_t tfull0 = smem_u32(bars + 2 * NS), tempty0 = smem_u32(bars + 2 * NS + 2);
  const uint32_t drain = smem_u32(bars + 2 * NS + 4);
  volatile int* abort_flag = (volatile int*)(bars + 2 * NS + 5);
  uint32_t* tmem_slot = (uint32_t*)(bars + 2 * NS + 6);
  const int rank = CG == 2 ? (int)cluster_ctarank() : 0;
  const bool leader = rank == 0;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      // rank 0 of a pair with gathered rows also counts the relay of rank 1's gathers
      mbar_init(full0 + 8 * s, (MD::kCpAsync ? kProducerWarps * 32 : 1) + (CG == 2 && leader && MD::kCpAsync ? 1 : 0));
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, CG == 2 ? 2 * kEpiWarps : MT * kEpiWarps * 32);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {
    if (CG == 2) {
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                   "r"(TMEM_COLS)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                   "r"(TMEM_COLS)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  if (CG == 2) cluster_sync();   // the peer's barriers are initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int ntiles = total_tiles<SCHED, CG, MT>(p);
  const int tile0 = blockIdx.x / CG, tstep = gridDim.x / CG;
  const uint32_t lead_full0 = CG == 2 ? mapa_shared(full0, 0) : full0;   // rank 0's full barriers

  if (warp < kProducerWarps) {
    // ------------------------------------------------------------ producers
    int it = 0;
    bool ok = true;
    for (int L = tile0; L < ntiles && ok; L += tstep) {
      const Tile t = map_tile<SCHED, CG, MT>(p, L, rank);
      const bf16* gsrc[8 * MT];
      uint32_t gbytes[8 * MT];
      if (AMODE == A_GATHER_K) {
#pragma unroll
        for (int j = 0; j < 8 * MT; ++j) {
          const int r = (j >> 3) * BM + warp * 32 + (j & 7) * 4 + (lane >> 3);
          const int row = t.row0 + r;
          const bool v = row < t.row_end;
          const int tok = v ? p.row_token[row] : 0;
          gsrc[j] = p.A + (size_t)tok * p.lda + (lane & 7) * 8;
          gbytes[j] = v ? 16u : 0u;
        }
      }
      // GATHER_MN: the token index of each gathered K row is loaded two blocks ahead so the L2
      // round trip overlaps the pipeline.
      constexpr bool kTokRing = AMODE == A_GATHER_MN || BMODE == B_GATHER_MN;
      int tk0 = 0, tk1 = 0, tk2 = 0;
      auto tok_at = [&](int kb) {
        // lane l < 16 of warp w: token of K row 16w + l of block kb
        const int row = t.row0 + kb * BK + 16 * warp + (lane & 15);
        return (kb < t.nkb && row < t.row_end) ? p.row_token[row] : 0;
      };
      if (kTokRing) {
        tk1 = tok_at(0);
        tk2 = tok_at(1);
      }
      for (int kb = t.kb0; kb < t.nkb; ++kb, ++it) {
        if (kTokRing) {
          tk0 = tk1;
          tk1 = tk2;
          tk2 = tok_at(kb + 2);
        }
        const int s = it % NS;
        const uint32_t ph = (it / NS) & 1;
        if (!mbar_wait(empty0 + 8 * s, ph ^ 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        const uint32_t sa = smem_u32(stage_base + s * SM::STAGE);
        const uint32_t sb = sa + SM::A_BYTES;
        load_stage<BN, AMODE, BMODE, SCHED, CG, MD::kCpAsync, MT>(p, &tmA, &tmB, t, kb, sa, sb, full0 + 8 * s, gsrc,
                                                                  gbytes, tk0, rank, lead_full0 + 8 * s);
        // the stage's full barrier counts this thread's arrival once all of its copies so far have
        // landed; the producer goes straight on to the next stage
        if (MD::kCpAsync) cp_async_mbar_arrive_noinc(full0 + 8 * s);
      }
    }
    if (MD::kCpAsync) cp_async_wait<0>();
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0 && CG == 2 && !leader && MD::kCpAsync) {
      // rank 1: relay each stage's gathered rows, once landed, to rank 0's full barrier
      int it = 0;
      bool ok = true;
      for (int L = tile0; L < ntiles && ok; L += tstep) {
        const Tile t = map_tile<SCHED, CG>(p, L, rank);
        for (int kb = t.kb0; kb < t.nkb; ++kb, ++it) {
          const int s = it % NS;
          if (!mbar_wait(full0 + 8 * s, (it / NS) & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          if (MD::kCpAsync) fence_proxy_async();   // cp.async (generic proxy) writes seen by the pair's MMA
          mbar_arrive_cluster(lead_full0 + 8 * s);
        }
      }
    } else if (lane == 0 && leader) {
      int it = 0, tcount = 0;
      bool ok = true;
      for (int L = tile0; L < ntiles && ok; L += tstep, ++tcount) {
        const Tile t = map_tile<SCHED, CG, MT>(p, L, rank);
        const int acc = tcount % NACC;
        const uint32_t aph = (tcount / NACC) & 1;
        if (!(CG == 2 ? mbar_wait_cluster(tempty0 + 8 * acc, aph ^ 1, abort_flag, p.status)
                      : mbar_wait(tempty0 + 8 * acc, aph ^ 1, abort_flag, p.status)))
          break;
        tc_fence_after();
        const uint32_t dcol = tmem_base + acc * BN;
        for (int kb = t.kb0; kb < t.nkb; ++kb, ++it) {
          const int s = it % NS;
          const uint32_t ph = (it / NS) & 1;
          if (!(CG == 2 && MD::kCpAsync ? mbar_wait_cluster(full0 + 8 * s, ph, abort_flag, p.status)
                                        : mbar_wait(full0 + 8 * s, ph, abort_flag, p.status))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (MD::kCpAsync) fence_proxy_async();   // cp.async (generic proxy) writes seen by the MMA
          const uint32_t sa = smem_u32(stage_base + s * SM::STAGE);
          const uint32_t sb = sa + SM::A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t da = MD::kAMn ? desc_mnmajor(sa + k * 2048) : desc_kmajor(sa + k * 32);
            const uint64_t db = MD::kBMn ? desc_mnmajor(sb + k * 2048) : desc_kmajor(sb + k * 32);
            if (CG == 2) mma_bf16_pair(dcol, da, db, IDESC, (kb > t.kb0 || k > 0) ? 1u : 0u);
            else mma_bf16(dcol, da, db, IDESC, (kb > t.kb0 || k > 0) ? 1u : 0u);
            if (MT == 2 && t.two)   // second 128-row tile: its own accumulator, the same B tile
              mma_bf16(dcol + BN, desc_kmajor(sa + BM * 128 + k * 32), db, IDESC, (kb > t.kb0 || k > 0) ? 1u : 0u);
          }
          if (CG == 2) mma_commit_pair_mc(empty0 + 8 * s, 0x3);
          else mma_commit(empty0 + 8 * s);
        }
        if (!ok) break;
        if (CG == 2) mma_commit_pair_mc(tfull0 + 8 * acc, 0x3);
        else mma_commit(tfull0 + 8 * acc);
      }
      // drain: wait until every issued MMA has completed before TMEM is freed
      if (CG == 2) mma_commit_pair(drain);
      else mma_commit(drain);
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(drain, 0)) {
        if (global_ns() - t0 > kWaitLimitNs) {
          set_error(p.status, MOE_ERR_TIMEOUT);
          break;
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp & 3;                  // TMEM lane quadrant of this warp: lanes 32*ew..
    const int half = MT == 2 && warp > kMmaWarp ? 1 : 0;   // MT = 2: which 128-row tile it drains
    const int r = half * BM + ew * 32 + lane;   // tile row
    int tcount = 0;
    for (int L = tile0; L < ntiles; L += tstep, ++tcount) {
      const Tile t = map_tile<SCHED, CG, MT>(p, L, rank);
      const int acc = tcount % NACC;
      const uint32_t aph = (tcount / NACC) & 1;
      if (!(CG == 2 ? mbar_wait_cluster(tfull0 + 8 * acc, aph, abort_flag, p.status)
                    : mbar_wait(tfull0 + 8 * acc, aph, abort_flag, p.status)))
        break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (acc + half) * BN + ((uint32_t)(ew * 32) << 16);
      const int row = t.row0 + r;   // SEG_M / DENSE output row
      const bool valid = row < t.row_end;
      if (MT == 2 && half && !t.two) {
        // the second tile holds no rows of the segment: nothing was accumulated for it
      } else if (EPI == EPI_SWIGLU) {
        epi_swiglu<BN>(p, t, tbase, row, valid);
      } else if (EPI == EPI_GATE || EPI == EPI_STORE) {
        epi_scale_store<BN, EPI == EPI_GATE>(p, t, tbase, row, valid);
      } else if (EPI == EPI_F32) {
        float* obase = p.ksplit > 1 ? p.part + (size_t)t.ks * p.dense_rows * p.ldo : (float*)p.out;
        float* orow = obase + (size_t)row * p.ldo + t.n * BN;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t a[32];
          tmem_ld32(tbase + c0, a);
          tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (t.n * BN + c0 + i < p.n_valid) orow[c0 + i] = __uint_as_float(a[i]);
          }
        }
      } else if (EPI == EPI_DH) {
        // r = dy_t Wd[e] for the BN features n*BN..: SwiGLU backward with the saved u, v, which
        // (like du, dv) sit in 128-feature blocks [u of block b | v of block b]; dg partials over
        // each 64-feature quarter. The last tile may run past f (its B columns were zero-filled):
        // blocks at or beyond f are skipped.
        static_assert(EPI != EPI_DH || BN % 128 == 0, "EPI_DH works on whole 128-feature blocks");
        const float g = valid ? p.row_gate[row] : 0.f;
        const bf16* uvrow = p.uv + (size_t)row * p.ld_uv;
        bf16* dudvrow = (bf16*)p.out + (size_t)row * p.ld_uv;
        bf16* hgrow = (bf16*)p.out2 + (size_t)row * p.ldo + t.n * BN;
        float dgp = 0.f;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          const int feat = t.n * BN + c0;   // first feature of this chunk
          if (feat >= p.ldo) break;
          const int blk = (feat >> 7) * 256 + (c0 & 127);   // column of u (v: + 128) in uv / dudv
          uint32_t a[32];
          tmem_ld32(tbase + c0, a);
          tmem_ld_wait();
          if (valid) {
            float uf[32], vf[32], du[32], dv[32], hg[32];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              unpack8_to(uvrow + blk + q * 8, uf + q * 8);
              unpack8_to(uvrow + blk + 128 + q * 8, vf + q * 8);
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float rr = __uint_as_float(a[i]);
              const float su = sigmoid_f(uf[i]);
              const float sl = uf[i] * su;
              const float hv = sl * vf[i];
              dgp = fmaf(rr, hv, dgp);
              const float dh = g * rr;
              du[i] = dh * vf[i] * su * (1.f + uf[i] * (1.f - su));
              dv[i] = dh * sl;
              hg[i] = g * hv;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              *reinterpret_cast<uint4*>(dudvrow + blk + q * 8) = pack8(du + q * 8);
              *reinterpret_cast<uint4*>(dudvrow + blk + 128 + q * 8) = pack8(dv + q * 8);
              *reinterpret_cast<uint4*>(hgrow + c0 + q * 8) = pack8(hg + q * 8);
            }
            if ((c0 & 63) == 32) {
              if (row < p.A_rows) p.dg_part[(size_t)row * p.dg_slots + (feat - 32) / 64] = dgp;
              dgp = 0.f;
            }
          }
        }
      } else {
        // Weight gradients (dW13, dWd): each warp writes its 32 rows of the tile as 32x64 sub-tiles
        // through a double-buffered 128-byte-swizzled staging buffer, stored by TMA.
        const bool empty = t.nkb == 0;
        const CUtensorMap* tmo = &tmC;
        // dW13: an M tile of 128 packed rows is all gate rows (m even, dWg) or all up rows (m odd,
        // dWu); dWd: one plane, and a last n-tile may run past the n_valid columns (its B columns
        // were zero-filled): sub-tiles at or beyond them are not stored
        if (EPI == EPI_DW13 && (t.m & 1)) tmo = &tmC2;
        const int orow0 = EPI == EPI_DW13 ? t.e * (p.m_tiles / 2) * BM + (t.m >> 1) * BM + ew * 32
                                          : (t.e * p.m_tiles + t.m) * BM + ew * 32;
        const uint32_t wbuf = smem_u32(out_stage) + ew * 2 * 4096;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 64) {
          const int sub = c0 >> 6;
          const uint32_t buf = wbuf + (sub & 1) * 4096;
          if (EPI == EPI_DWD && t.n * BN + c0 >= p.n_valid) break;
          float of[64];
          if (!empty) {
            uint32_t a[32], b[32];
            tmem_ld32(tbase + c0, a);
            tmem_ld32(tbase + c0 + 32, b);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              of[i] = __uint_as_float(a[i]);
              of[32 + i] = __uint_as_float(b[i]);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 64; ++i) of[i] = 0.f;
          }
          if (p.accumulate) {
            const bf16* base = (EPI == EPI_DW13 && (t.m & 1)) ? (const bf16*)p.out2 : (const bf16*)p.out;
            const bf16* old = base + (size_t)(orow0 + lane) * p.ldo + t.n * BN + c0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              float o8[8];
              unpack8(*reinterpret_cast<const uint4*>(old + q * 8), o8);
#pragma unroll
              for (int i = 0; i < 8; ++i) of[q * 8 + i] += o8[i];
            }
          }
          // the store that last read this buffer (two sub-tiles ago) must have finished reading it
          if (lane == 0) bulk_wait_read<1>();
          __syncwarp();
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint4 v = pack8(of + q * 8);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(buf + lane * 128 + ((q ^ (lane & 7)) << 4)),
                         "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                         : "memory");
          }
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d_hint(tmo, t.n * BN + c0, orow0, buf, policy_evict_first());
            bulk_commit();
          }
        }
      }
      tc_fence_before();
      if (CG == 2) {
        // one arrival per epilogue warp of either CTA, on rank 0's barrier
        __syncwarp();
        if (lane == 0) {
          if (leader) mbar_arrive(tempty0 + 8 * acc);
          else mbar_arrive_cluster(mapa_shared(tempty0 + 8 * acc, 0));
        }
      } else {
        mbar_arrive(tempty0 + 8 * acc);
      }
    }
  }
  if (SCHED == SCHED_SEG_K && warp >= kProducerWarps && warp < kMmaWarp && lane == 0) bulk_wait<0>();
  tc_fence_before();
  __syncthreads();
  if (CG == 2) cluster_sync();   // neither CTA leaves while the pair's MMAs or arrivals may touch it
  if (warp == kMmaWarp) {
    tc_fence_after();
    if (CG == 2)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                   : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                   : "memory");
  }
}

// ------------------------------------------------------- fused expert kernel
// The forward's two expert GEMMs in one persistent launch: the gate/up tiles, then the down tiles,
// taken from one static order (CTA b takes entries b, b + grid, ...), so a CTA that runs out of
// gate/up tiles goes straight on to down tiles instead of idling through the gate/up tail and a
// kernel boundary. A down tile of (segment e, m-tile m) needs the h rows that all gate/up tiles of
// (e, m) write: each epilogue warp of a gate/up tile adds 1 to dep[mt_off[e] + m] once its rows
// are stored (and to done[2]), and the producer issuing the down tile's loads waits (acquire,
// bounded) for kEpiWarps x gate/up n-tiles arrivals, or sees done[2] complete. Every dependency
// points to an earlier entry of the order and every CTA walks its entries in increasing order, so
// with all CTAs resident (cooperative launch) the waits end. The last CTA to finish (ticket
// done[1]) zeroes the counters for the next call. Every wait gives up after kWaitLimitNs with
// MOE_ERR_TIMEOUT.
struct FusedParams {
  TcParams gu, dn;       // gate/up and down GEMMs, as for the separate kernels
  unsigned* dep;         // per m-tile of the segment schedule
  unsigned* done;        // [1]: CTAs finished; [2]: gate/up-tile epilogue warps finished
};

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Waits until *p >= need; false (status set) after kWaitLimitNs or once this CTA aborted.
__device__ __noinline__ bool wait_count(const unsigned* p, unsigned need, volatile int* abort_flag, int* status) {
  if (ld_acquire_u32(p) >= need) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    __nanosleep(128);
    if (ld_acquire_u32(p) >= need) return true;
    if ((i & 15) == 0) {
      if (*abort_flag) return false;
      if (global_ns() - t0 > kWaitLimitNs) {
        set_error(status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// One warp's arrival on a counter after its global stores (read by other CTAs' TMA loads).
__device__ __forceinline__ void signal_count(unsigned* p, int lane) {
  fence_proxy_async_global();
  __syncwarp();
  if (lane == 0) {
    __threadfence();
    atomicAdd(p, 1u);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    fused_experts_kernel(const __grid_constant__ CUtensorMap tmW13, const __grid_constant__ CUtensorMap tmH,
                         const __grid_constant__ CUtensorMap tmWd, const __grid_constant__ FusedParams q) {
  constexpr int BN = 256;
  using SM = Smem<BN, SCHED_SEG_M, 1>;
  constexpr int NS = SM::NS;
  constexpr uint32_t TMEM_COLS = 512;
  constexpr uint32_t IDESC = idesc_bf16(BM, BN, 0, 0);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* stage_base = smem;
  uint64_t* bars = (uint64_t*)(smem + NS * SM::STAGE);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + NS);
  const uint32_t tfull0 = smem_u32(bars + 2 * NS), tempty0 = smem_u32(bars + 2 * NS + 2);
  const uint32_t drain = smem_u32(bars + 2 * NS + 4);
  volatile int* abort_flag = (volatile int*)(bars + 2 * NS + 5);
  uint32_t* tmem_slot = (uint32_t*)(bars + 2 * NS + 6);
  int* ticket = (int*)(bars + 2 * NS + 7);
  int* status = q.gu.status;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full0 + 8 * s, kProducerWarps * 32);   // every producer thread arrives on every stage
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, kEpiWarps * 32);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int n_gu = total_tiles<SCHED_SEG_M, 1>(q.gu);
  const int n_all = n_gu + total_tiles<SCHED_SEG_M, 1>(q.dn);
  const unsigned gu_arrivals = kEpiWarps * q.gu.n_tiles;   // per m-tile

  if (warp < kProducerWarps) {
    // ------------------------------------------------------------ producers
    int it = 0;
    bool ok = true;
    bool all_up = false;   // every gate/up tile finished: no down tile needs to wait any more
    for (int G = blockIdx.x; G < n_all && ok; G += gridDim.x) {
      const bool up = G < n_gu;
      const Tile t = up ? map_tile<SCHED_SEG_M, 1>(q.gu, G, 0) : map_tile<SCHED_SEG_M, 1>(q.dn, G - n_gu, 0);
      const bf16* gsrc[8];
      uint32_t gbytes[8];
      if (up) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int r = warp * 32 + j * 4 + (lane >> 3);
          const int row = t.row0 + r;
          const bool v = row < t.row_end;
          const int tok = v ? q.gu.row_token[row] : 0;
          gsrc[j] = q.gu.A + (size_t)tok * q.gu.lda + (lane & 7) * 8;
          gbytes[j] = v ? 16u : 0u;
        }
      } else if (threadIdx.x == 0 && !all_up) {
        // the h rows of this m-tile: every gate/up tile of (e, m) finished by all its epilogue warps
        if (ld_acquire_u32(q.done + 2) >= kEpiWarps * (unsigned)n_gu) all_up = true;
        else if (!wait_count(q.dep + q.gu.mt_off[t.e] + t.m, gu_arrivals, abort_flag, status)) ok = false;
        fence_proxy_async_global();
      }
      for (int kb = 0; kb < t.nkb && ok; ++kb, ++it) {
        const int s = it % NS;
        const uint32_t ph = (it / NS) & 1;
        if (!mbar_wait(empty0 + 8 * s, ph ^ 1, abort_flag, status)) {
          ok = false;
          break;
        }
        const uint32_t sa = smem_u32(stage_base + s * SM::STAGE);
        const uint32_t sb = sa + SM::A_BYTES;
        if (up)
          load_stage<BN, A_GATHER_K, B_TMA_K, SCHED_SEG_M, 1, true>(q.gu, &tmW13, &tmW13, t, kb, sa, sb,
                                                                     full0 + 8 * s, gsrc, gbytes, 0, 0, 0);
        else
          load_stage<BN, A_TMA_K, B_TMA_K, SCHED_SEG_M, 1, true>(q.dn, &tmH, &tmWd, t, kb, sa, sb, full0 + 8 * s,
                                                                  gsrc, gbytes, 0, 0, 0);
        cp_async_mbar_arrive_noinc(full0 + 8 * s);
      }
    }
    cp_async_wait<0>();
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      int it = 0, tcount = 0;
      bool ok = true;
      for (int G = blockIdx.x; G < n_all && ok; G += gridDim.x, ++tcount) {
        const bool up = G < n_gu;
        const Tile t = up ? map_tile<SCHED_SEG_M, 1>(q.gu, G, 0) : map_tile<SCHED_SEG_M, 1>(q.dn, G - n_gu, 0);
        const int acc = tcount & 1;
        if (!mbar_wait(tempty0 + 8 * acc, ((tcount >> 1) & 1) ^ 1, abort_flag, status)) break;
        tc_fence_after();
        const uint32_t dcol = tmem_base + acc * BN;
        for (int kb = 0; kb < t.nkb; ++kb, ++it) {
          const int s = it % NS;
          if (!mbar_wait(full0 + 8 * s, (it / NS) & 1, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (up) fence_proxy_async();   // gathered rows (cp.async, generic proxy) seen by the MMA
          const uint32_t sa = smem_u32(stage_base + s * SM::STAGE);
          const uint32_t sb = sa + SM::A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma_bf16(dcol, desc_kmajor(sa + k * 32), desc_kmajor(sb + k * 32), IDESC, (kb > 0 || k > 0) ? 1u : 0u);
          mma_commit(empty0 + 8 * s);
        }
        if (!ok) break;
        mma_commit(tfull0 + 8 * acc);
      }
      mma_commit(drain);
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(drain, 0)) {
        if (global_ns() - t0 > kWaitLimitNs) {
          set_error(status, MOE_ERR_TIMEOUT);
          break;
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - kProducerWarps;
    const int r = ew * 32 + lane;
    int tcount = 0;
    for (int G = blockIdx.x; G < n_all; G += gridDim.x, ++tcount) {
      const bool up = G < n_gu;
      const Tile t = up ? map_tile<SCHED_SEG_M, 1>(q.gu, G, 0) : map_tile<SCHED_SEG_M, 1>(q.dn, G - n_gu, 0);
      const int acc = tcount & 1;
      if (!mbar_wait(tfull0 + 8 * acc, (tcount >> 1) & 1, abort_flag, status)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + acc * BN + ((uint32_t)(ew * 32) << 16);
      const int row = t.row0 + r;
      const bool valid = row < t.row_end;
      if (up) {
        epi_swiglu<BN>(q.gu, t, tbase, row, valid);
        signal_count(q.dep + q.gu.mt_off[t.e] + t.m, lane);
        if (lane == 0) atomicAdd(q.done + 2, 1u);
      } else {
        epi_scale_store<BN, true>(q.dn, t, tbase, row, valid);
      }
      tc_fence_before();
      mbar_arrive(tempty0 + 8 * acc);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                 : "memory");
  }
  // the last CTA to finish zeroes the counters for the next call
  if (threadIdx.x == 0) {
    __threadfence();
    *ticket = (int)atomicAdd(q.done + 1, 1u);
  }
  __syncthreads();
  if (*ticket == (int)gridDim.x - 1) {
    __threadfence();
    const int nm = q.gu.mt_off[q.gu.nseg];
    for (int i = threadIdx.x; i < nm; i += blockDim.x) q.dep[i] = 0;
    __syncthreads();
    if (threadIdx.x == 0) {
      q.done[1] = 0;
      q.done[2] = 0;
      __threadfence();
    }
  }
}

// ------------------------------------------------------ whole-forward kernel
// The whole forward in one cooperative persistent launch: router logits (tcgen05 tiles, the same
// K splits as the separate router launch, partials added in split order), top-k and gates, the
// chunk histograms, the scan (one CTA), the stable permutation, the gate/up and down GEMM tiles,
// and the combine. Phases are separated by grid-wide barriers; every wait (barrier, dependency
// counter, mbarrier) is bounded and past its limit records MOE_ERR_TIMEOUT, raises a global abort
// word that every CTA's later waits see, and the kernel runs to its end without further work.
// The expert tiles come from a device tile queue (an atomic head, gate/up tiles first): the
// producer's first thread takes the next tile and publishes it in a small shared-memory ring that
// the producer warps, the MMA thread and the epilogue warps read in order; a down tile's loads
// wait for the h rows of its row block (per-row-block counters, as in fused_experts_kernel).
// Dependencies point only to tiles taken earlier, and every CTA finishes its tiles in the order it
// took them, so with all CTAs resident (cooperative launch) every wait ends. Each output element
// is computed with the same instructions in the same order as the separate launches: results are
// bit-identical to them. The last CTA to finish zeroes the counters for the next call.
struct FwdParams {
  TcParams rt, gu, dn;   // router (DENSE, EPI_F32: partials in rt.part when rt.ksplit > 1), gate/up, down
  const float* bias;
  float* logits;         // [T, E]
  int* idx;              // [T, k]
  float* gate;           // [T, k]
  int* chunk_hist;
  int* chunk_base;
  int* cnt;
  int* off;
  int* mt_off;
  int* perm;
  int* inv;
  int* row_token;
  float* row_gate;
  const bf16* o;         // gated expert outputs [R, d] (written by the down tiles)
  bf16* y;               // [T, d]
  int T, E, S, k, d, router, renorm, A, nch;
  float scale;
  unsigned* dep;         // per m-tile arrival counters
  int dep_len;           // their number (cleared in full after every call)
  unsigned* ctr;         // [0] tile queue head, [1] CTAs finished, [2] gate/up epilogue warps finished,
                         // [3] grid-barrier arrivals, [4] abort
};

constexpr int kTq = 32;   // entries of the shared tile-queue ring
constexpr int kFwdScratch = permute_smem(kThreads / 32) > kScanSmem ? permute_smem(kThreads / 32) : kScanSmem;
// ring, then the SIMT scratch and the queue ring, then the barriers (aligned to 8) and two ints
constexpr int kFwdSmem = Smem<256, SCHED_SEG_M, 1>::NS * Smem<256, SCHED_SEG_M, 1>::STAGE + 4 * (kFwdScratch + 2 * kTq) +
                         8 + 8 * (2 * Smem<256, SCHED_SEG_M, 1>::NS + 8) + 1024;
static_assert(kFwdSmem <= kSmemMax, "whole-forward kernel shared memory");

// Grid-wide barrier number gen (1, 2, ...): every CTA adds one to ctr[3] and waits until it reaches
// gen * gridDim.x. False (for the whole CTA) if the global abort word is raised or the wait passes
// kWaitLimitNs (then MOE_ERR_TIMEOUT is recorded and the abort word raised).
__device__ __noinline__ bool grid_barrier(unsigned* ctr, unsigned gen, int* status, int* ok_s) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(ctr + 3, 1u);
    const unsigned need = gen * gridDim.x;
    int ok = 1;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0; ld_acquire_u32(ctr + 3) < need; ++i) {
      __nanosleep(64);
      if ((i & 15) == 15) {
        if (ld_acquire_u32(ctr + 4)) {
          ok = 0;
          break;
        }
        if (global_ns() - t0 > kWaitLimitNs) {
          set_error(status, MOE_ERR_TIMEOUT);
          atomicExch(ctr + 4, 1u);
          ok = 0;
          break;
        }
      }
    }
    if (ok && ld_acquire_u32(ctr + 4)) ok = 0;
    __threadfence();
    *ok_s = ok;
  }
  __syncthreads();
  return *ok_s != 0;
}

__global__ void __launch_bounds__(kThreads, 1)
    fused_forward_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmWr,
                         const __grid_constant__ CUtensorMap tmW13, const __grid_constant__ CUtensorMap tmH,
                         const __grid_constant__ CUtensorMap tmWd, const __grid_constant__ FwdParams q) {
  constexpr int BN = 256;
  using SM = Smem<BN, SCHED_SEG_M, 1>;
  constexpr int NS = SM::NS;
  constexpr uint32_t TMEM_COLS = 512;
  constexpr uint32_t IDESC = idesc_bf16(BM, BN, 0, 0);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* stage_base = smem;
  int* scratch = (int*)(smem + NS * SM::STAGE);                     // SIMT phases
  volatile int* tq_tile = (volatile int*)(scratch + kFwdScratch);   // [kTq] tile of queue entry i
  volatile int* tq_seq = tq_tile + kTq;                              // [kTq] entry number held
  uint64_t* bars = (uint64_t*)(((uintptr_t)(scratch + kFwdScratch + 2 * kTq) + 7) & ~(uintptr_t)7);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + NS);
  const uint32_t tfull0 = smem_u32(bars + 2 * NS), tempty0 = smem_u32(bars + 2 * NS + 2);
  const uint32_t drain = smem_u32(bars + 2 * NS + 4);
  volatile int* abort_flag = (volatile int*)(bars + 2 * NS + 5);
  uint32_t* tmem_slot = (uint32_t*)(bars + 2 * NS + 6);
  int* ticket = (int*)(bars + 2 * NS + 7);
  int* ok_s = ticket + 1;
  int* status = q.gu.status;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full0 + 8 * s, kProducerWarps * 32);   // every producer thread arrives on every stage
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, kEpiWarps * 32);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int i = threadIdx.x; i < kTq; i += blockDim.x) tq_seq[i] = -1;
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // pipeline positions, kept by each role across the two GEMM phases
  int it = 0, tcount = 0;
  bool ok = true;   // this thread's role has seen no failed wait

  // ------------------------------------------------------------- phase 1: router logit tiles
  const int n_rt = total_tiles<SCHED_DENSE, 1>(q.rt);
  if (warp < kProducerWarps) {
    const bf16* gsrc[8] = {};
    uint32_t gbytes[8] = {};
    for (int L = blockIdx.x; L < n_rt && ok; L += gridDim.x) {
      const Tile t = map_tile<SCHED_DENSE, 1>(q.rt, L, 0);
      for (int kb = t.kb0; kb < t.nkb; ++kb, ++it) {
        const int s = it % NS;
        if (!mbar_wait(empty0 + 8 * s, ((it / NS) & 1) ^ 1, abort_flag, status)) {
          ok = false;
          break;
        }
        const uint32_t sa = smem_u32(stage_base + s * SM::STAGE);
        load_stage<BN, A_TMA_K, B_TMA_K, SCHED_DENSE, 1, true>(q.rt, &tmX, &tmWr, t, kb, sa, sa + SM::A_BYTES,
                                                              full0 + 8 * s, gsrc, gbytes, 0, 0, 0);
        cp_async_mbar_arrive_noinc(full0 + 8 * s);
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      for (int L = blockIdx.x; L < n_rt && ok; L += gridDim.x, ++tcount) {
        const Tile t = map_tile<SCHED_DENSE, 1>(q.rt, L, 0);
        const int acc = tcount & 1;
        if (!mbar_wait(tempty0 + 8 * acc, ((tcount >> 1) & 1) ^ 1, abort_flag, status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dcol = tmem_base + acc * BN;
        for (int kb = t.kb0; kb < t.nkb; ++kb, ++it) {
          const int s = it % NS;
          if (!mbar_wait(full0 + 8 * s, (it / NS) & 1, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(stage_base + s * SM::STAGE);
          const uint32_t sb = sa + SM::A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma_bf16(dcol, desc_kmajor(sa + k * 32), desc_kmajor(sb + k * 32), IDESC,
                     (kb > t.kb0 || k > 0) ? 1u : 0u);
          mma_commit(empty0 + 8 * s);
        }
        if (!ok) break;
        mma_commit(tfull0 + 8 * acc);
      }
    }
    __syncwarp();
  } else {
    const int ew = warp - kProducerWarps;
    const int r = ew * 32 + lane;
    for (int L = blockIdx.x; L < n_rt && ok; L += gridDim.x, ++tcount) {
      const Tile t = map_tile<SCHED_DENSE, 1>(q.rt, L, 0);
      const int acc = tcount & 1;
      if (!mbar_wait(tfull0 + 8 * acc, (tcount >> 1) & 1, abort_flag, status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + acc * BN + ((uint32_t)(ew * 32) << 16);
      const int row = t.row0 + r;
      const bool valid = row < t.row_end;
      float* obase = q.rt.ksplit > 1 ? q.rt.part + (size_t)t.ks * q.rt.dense_rows * q.rt.ldo : (float*)q.rt.out;
      float* orow = obase + (size_t)row * q.rt.ldo + t.n * BN;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t a[32];
        tmem_ld32(tbase + c0, a);
        tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (t.n * BN + c0 + i < q.rt.n_valid) orow[c0 + i] = __uint_as_float(a[i]);
        }
      }
      tc_fence_before();
      mbar_arrive(tempty0 + 8 * acc);
    }
  }
  if (!ok) {
    *abort_flag = 1;
    atomicExch(q.ctr + 4, 1u);
  }

  // --------------------------------------------- phases 2-6: the routing, CTA- or warp-parallel
  const int gwarp = blockIdx.x * (kThreads / 32) + warp, nwarps = gridDim.x * (kThreads / 32);
  bool live = grid_barrier(q.ctr, 1, status, ok_s);
  if (live && q.rt.ksplit > 1) {
    // logits = the K splits' partials added in split order
    const long n = (long)q.T * q.E;
    for (long i = (long)blockIdx.x * kThreads + threadIdx.x; i < n; i += (long)gridDim.x * kThreads) {
      float sum = 0.f;
      for (int ks = 0; ks < q.rt.ksplit; ++ks) sum += __ldcg(q.rt.part + ks * n + i);
      q.logits[i] = sum;
    }
  }
  live = grid_barrier(q.ctr, 2, status, ok_s) && live;
  if (live)
    for (int t = gwarp; t < q.T; t += nwarps)
      warp_topk_gates(q.logits + (size_t)t * q.E, q.bias, q.E, q.k, q.router, q.renorm, q.scale,
                      q.idx + (size_t)t * q.k, q.gate + (size_t)t * q.k);
  live = grid_barrier(q.ctr, 3, status, ok_s) && live;
  if (live)
    for (int ch = blockIdx.x; ch < q.nch; ch += gridDim.x) hist_chunk(q.idx, q.A, q.E, ch, q.chunk_hist, status, scratch);
  live = grid_barrier(q.ctr, 4, status, ok_s) && live;
  if (live && blockIdx.x == 0)
    scan_segments(q.chunk_hist, q.nch, q.E, q.S, q.T, q.chunk_base, q.cnt, q.off, q.mt_off, scratch);
  live = grid_barrier(q.ctr, 5, status, ok_s) && live;
  if (live) {
    for (int ch = blockIdx.x; ch < q.nch; ch += gridDim.x)
      permute_chunk(q.idx, q.gate, q.A, q.E, q.k, ch, q.chunk_base, q.perm, q.inv, q.row_token, q.row_gate, scratch);
    if (q.S)
      for (int t = blockIdx.x * kThreads + threadIdx.x; t < q.T; t += gridDim.x * kThreads) {
        q.row_token[q.A + t] = t;
        q.row_gate[q.A + t] = 1.0f;
      }
  }
  live = grid_barrier(q.ctr, 6, status, ok_s) && live;
  if (!live) *abort_flag = 1;

  // -------------------------------------------------- phase 7: expert tiles from the tile queue
  const int n_gu = live ? total_tiles<SCHED_SEG_M, 1>(q.gu) : 0;
  const int n_all = live ? n_gu + total_tiles<SCHED_SEG_M, 1>(q.dn) : 0;
  const unsigned gu_arrivals = kEpiWarps * q.gu.n_tiles;   // per m-tile
  // queue entry i of this CTA: waits until published (bounded), -1 past the last tile or on abort.
  // The publishing thread is at most a few tiles ahead of any reader (its loads wait for stages the
  // MMA freed, the MMA waits for accumulators the epilogue freed), far less than kTq.
  auto entry = [&](int i) -> int {
    const int slot = i % kTq;
    const uint64_t t0 = global_ns();
    for (uint32_t n = 0; tq_seq[slot] != i; ++n) {
      if ((n & 63) == 63) {
        if (*abort_flag) return -1;
        if (global_ns() - t0 > kWaitLimitNs) {
          set_error(status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          return -1;
        }
      }
    }
    __threadfence_block();
    return tq_tile[slot];
  };
  if (warp < kProducerWarps) {
    bool all_up = false;   // every gate/up tile finished: no down tile needs to wait any more
    for (int i = 0; live && ok; ++i) {
      int G;
      if (threadIdx.x == 0) {
        const int G0 = *abort_flag ? n_all : (int)atomicAdd(q.ctr + 0, 1u);
        G = G0 < n_all ? G0 : -1;
        tq_tile[i % kTq] = G;
        __threadfence_block();
        tq_seq[i % kTq] = i;
      } else {
        G = entry(i);
      }
      if (G < 0) break;
      const bool up = G < n_gu;
      const Tile t = up ? map_tile<SCHED_SEG_M, 1>(q.gu, G, 0) : map_tile<SCHED_SEG_M, 1>(q.dn, G - n_gu, 0);
      const bf16* gsrc[8];
      uint32_t gbytes[8];
      if (up) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int rr = warp * 32 + j * 4 + (lane >> 3);
          const int row = t.row0 + rr;
          const bool v = row < t.row_end;
          const int tok = v ? q.gu.row_token[row] : 0;
          gsrc[j] = q.gu.A + (size_t)tok * q.gu.lda + (lane & 7) * 8;
          gbytes[j] = v ? 16u : 0u;
        }
      } else if (threadIdx.x == 0 && !all_up) {
        // the h rows of this m-tile: every gate/up tile of (e, m) finished by all its epilogue warps
        if (ld_acquire_u32(q.ctr + 2) >= kEpiWarps * (unsigned)n_gu) all_up = true;
        else if (!wait_count(q.dep + q.gu.mt_off[t.e] + t.m, gu_arrivals, abort_flag, status)) ok = false;
        fence_proxy_async_global();
      }
      for (int kb = 0; kb < t.nkb && ok; ++kb, ++it) {
        const int s = it % NS;
        if (!mbar_wait(empty0 + 8 * s, ((it / NS) & 1) ^ 1, abort_flag, status)) {
          ok = false;
          break;
        }
        const uint32_t sa = smem_u32(stage_base + s * SM::STAGE);
        const uint32_t sb = sa + SM::A_BYTES;
        if (up)
          load_stage<BN, A_GATHER_K, B_TMA_K, SCHED_SEG_M, 1, true>(q.gu, &tmW13, &tmW13, t, kb, sa, sb,
                                                                     full0 + 8 * s, gsrc, gbytes, 0, 0, 0);
        else
          load_stage<BN, A_TMA_K, B_TMA_K, SCHED_SEG_M, 1, true>(q.dn, &tmH, &tmWd, t, kb, sa, sb, full0 + 8 * s,
                                                                  gsrc, gbytes, 0, 0, 0);
        cp_async_mbar_arrive_noinc(full0 + 8 * s);
      }
    }
    cp_async_wait<0>();
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      for (int i = 0; live && ok; ++i, ++tcount) {
        const int G = entry(i);
        if (G < 0) break;
        const bool up = G < n_gu;
        const Tile t = up ? map_tile<SCHED_SEG_M, 1>(q.gu, G, 0) : map_tile<SCHED_SEG_M, 1>(q.dn, G - n_gu, 0);
        const int acc = tcount & 1;
        if (!mbar_wait(tempty0 + 8 * acc, ((tcount >> 1) & 1) ^ 1, abort_flag, status)) break;
        tc_fence_after();
        const uint32_t dcol = tmem_base + acc * BN;
        for (int kb = 0; kb < t.nkb; ++kb, ++it) {
          const int s = it % NS;
          if (!mbar_wait(full0 + 8 * s, (it / NS) & 1, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (up) fence_proxy_async();   // gathered rows (cp.async, generic proxy) seen by the MMA
          const uint32_t sa = smem_u32(stage_base + s * SM::STAGE);
          const uint32_t sb = sa + SM::A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma_bf16(dcol, desc_kmajor(sa + k * 32), desc_kmajor(sb + k * 32), IDESC, (kb > 0 || k > 0) ? 1u : 0u);
          mma_commit(empty0 + 8 * s);
        }
        if (!ok) break;
        mma_commit(tfull0 + 8 * acc);
      }
      // drain: wait until every issued MMA has completed before TMEM is freed
      mma_commit(drain);
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(drain, 0)) {
        if (global_ns() - t0 > kWaitLimitNs) {
          set_error(status, MOE_ERR_TIMEOUT);
          break;
        }
      }
    }
    __syncwarp();
  } else {
    const int ew = warp - kProducerWarps;
    const int r = ew * 32 + lane;
    for (int i = 0; live; ++i, ++tcount) {
      const int G = entry(i);
      if (G < 0) break;
      const bool up = G < n_gu;
      const Tile t = up ? map_tile<SCHED_SEG_M, 1>(q.gu, G, 0) : map_tile<SCHED_SEG_M, 1>(q.dn, G - n_gu, 0);
      const int acc = tcount & 1;
      if (!mbar_wait(tfull0 + 8 * acc, (tcount >> 1) & 1, abort_flag, status)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + acc * BN + ((uint32_t)(ew * 32) << 16);
      const int row = t.row0 + r;
      const bool valid = row < t.row_end;
      if (up) {
        epi_swiglu<BN>(q.gu, t, tbase, row, valid);
        signal_count(q.dep + q.gu.mt_off[t.e] + t.m, lane);
        if (lane == 0) atomicAdd(q.ctr + 2, 1u);
      } else {
        epi_scale_store<BN, true>(q.dn, t, tbase, row, valid);
      }
      tc_fence_before();
      mbar_arrive(tempty0 + 8 * acc);
    }
  }
  if (*abort_flag) atomicExch(q.ctr + 4, 1u);

  // ------------------------------------------------------------------- phase 8: the combine
  // y[t] = o[A + t] (shared) + sum_j o[inv[t k + j]], fp32 in that order, one rounding
  live = grid_barrier(q.ctr, 7, status, ok_s) && live;
  if (live) {
    const int vecs = q.d / 8;
    const long n = (long)q.T * vecs;
    for (long v = (long)blockIdx.x * kThreads + threadIdx.x; v < n; v += (long)gridDim.x * kThreads) {
      const int t = (int)(v / vecs), c = (int)(v % vecs) * 8;
      // all k + 1 rows in flight before the sum (nine warps per SM: the loads' latency must overlap)
      int rj[kMaxK];
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) rj[j] = j < q.k ? q.inv[(long)t * q.k + j] : 0;
      const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
      const uint4 us = q.S ? __ldcg(reinterpret_cast<const uint4*>(q.o + (long)(q.A + t) * q.d + c)) : zero;
      uint4 uj[kMaxK];
#pragma unroll
      for (int j = 0; j < kMaxK; ++j)
        uj[j] = j < q.k ? __ldcg(reinterpret_cast<const uint4*>(q.o + (long)rj[j] * q.d + c)) : zero;
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      auto add = [&](const uint4& u) {
        float f[8];
        unpack8(u, f);
#pragma unroll
        for (int w = 0; w < 8; ++w) acc[w] += f[w];
      };
      if (q.S) add(us);
#pragma unroll
      for (int j = 0; j < kMaxK; ++j)
        if (j < q.k) add(uj[j]);
      *reinterpret_cast<uint4*>(q.y + (long)t * q.d + c) = pack8(acc);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                 : "memory");
  }
  // the last CTA to finish zeroes the counters for the next call
  if (threadIdx.x == 0) {
    __threadfence();
    *ticket = (int)atomicAdd(q.ctr + 1, 1u);
  }
  __syncthreads();
  if (*ticket == (int)gridDim.x - 1) {
    __threadfence();
    for (int i = threadIdx.x; i < q.dep_len; i += blockDim.x) q.dep[i] = 0;
    __syncthreads();
    if (threadIdx.x == 0) {
      q.ctr[0] = 0;
      q.ctr[1] = 0;
      q.ctr[2] = 0;
      q.ctr[3] = 0;
      q.ctr[4] = 0;
      __threadfence();
    }
  }
}

// -------------------------------------------------------------- host side
template <int BN, int AMODE, int BMODE, int SCHED, int EPI, int CG = 1, int MT = 1>
cudaError_t launch(const CUtensorMap& tmA, const CUtensorMap& tmB, const TcParams& p, int grid, cudaStream_t s,
                   const CUtensorMap* tmC = nullptr, const CUtensorMap* tmC2 = nullptr) {
  auto kern = tc_gemm_kernel<BN, AMODE, BMODE, SCHED, EPI, CG, MT>;
  const int smem = Smem<BN, SCHED, CG, MT>::TOTAL;
  static bool attr = false;
  static int pair_grid = 0;   // CTAs of as many 2-CTA clusters as fit on the GPU at once
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  if (CG == 1) {
    MOE_TRY(launch_pdl(kern, dim3(grid), dim3(threads_for(MT)), smem, s, tmA, tmB, tmC ? *tmC : tmA,
        tmC2 ? *tmC2 : tmA, p));
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (!pair_grid) {
    cfg.gridDim = dim3(2 * (grid / 2));
    int clusters = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (clusters < 1) return cudaErrorInvalidConfiguration;
    pair_grid = 2 * clusters;
  }
  // persistent: never more clusters than run at once (a second wave would serialise the tail)
  cfg.gridDim = dim3(pair_grid < grid ? pair_grid : 2 * (grid / 2));
  return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmC ? *tmC : tmA, tmC2 ? *tmC2 : tmA, p);
}

constexpr int kBNup = 256;     // gate/up: 128 gate + 128 up columns
constexpr int kBNdown = 256;
constexpr int kBNrouter = 256;
constexpr int kBNdh = 256;     // two 128-feature blocks per tile (the last may hold one)
constexpr int kBNdx = 256;
constexpr int kBNdw13 = 256;
constexpr int kBNdwd = 256;

// CTA pairs are opt-in: on GB300 they measured no faster than single CTAs for these GEMMs (a
// segment with an odd tile count also computes an empty second tile), and the relay of gathered
// rows to rank 0 costs a cluster-scope release per stage.
bool use_pairs(const Layer& L, const Bufs&) { return L.pairs == 1; }
// Two 128-row tiles per CTA for the segment GEMMs over token rows (gate/up, down, dY.Wd, dx).
bool use_mt2(const Layer& L) { return L.row_tiles == 2 && L.pairs != 1; }
TcParams base_params(const Layer& L, const Bufs& B) {
  TcParams p = {};
  p.row_token = B.row_token;
  p.off = B.off;
  p.mt_off = B.mt_off;
  p.mp_off = B.mt_off + (L.E + L.S + 1);   // the routing scan stores the pair prefix after mt_off
  p.nseg = L.E + L.S;
  p.pstride = L.E + L.S + 1;
  p.A_rows = B.A;
  p.status = L.status;
  return p;
}

}  // namespace

bool tc_router_supported(const Layer& L) {
  return L.prec != MOE_FP32 && L.d % 64 == 0 && L.E <= kBNrouter && encode_fn() != nullptr;
}

bool tc_supported(const Layer& L) {
  return L.prec == MOE_BF16 && L.d % 256 == 0 && L.f % kGate == 0 && L.G == kGate && L.E <= kBNrouter &&
         encode_fn() != nullptr;
}

cudaError_t tc_init(Layer& L) {
  const uint64_t nseg = L.E + L.S;
  if (!make_tmap(&L.tm_W13, L.W13, L.d, nseg * 2 * L.f, BK, kBNup)) return cudaErrorInvalidValue;
  if (!make_tmap(&L.tm_Wd, L.Wd, L.f, nseg * L.d, BK, kBNdown)) return cudaErrorInvalidValue;
  if (!make_tmap(&L.tm_W13_mn, L.W13, L.d, nseg * 2 * L.f, 64, BK)) return cudaErrorInvalidValue;
  if (!make_tmap(&L.tm_Wd_mn, L.Wd, L.f, nseg * L.d, 64, BK)) return cudaErrorInvalidValue;
  if (!make_tmap(&L.tm_W13_h, L.W13, L.d, nseg * 2 * L.f, BK, kBNup / 2)) return cudaErrorInvalidValue;
  if (!make_tmap(&L.tm_Wd_h, L.Wd, L.f, nseg * L.d, BK, kBNdown / 2)) return cudaErrorInvalidValue;
  return cudaSuccess;
}

// K splits of the router GEMM: with few row tiles (small T) about one CTA per SM gets work (at
// least 4 K blocks per split, at most 16 splits). A function of the shapes only, so that every
// routing call (route, forward, the no-allocation route) sums the logits in the same order; the
// partials must fit kRouterPartBytes and the forward scratch o (R x d x 2 bytes).
int tc_router_splits(const Layer& L, int T) {
  const int tiles = (T + BM - 1) / BM;
  const int nk = L.d / BK;
  int ks = L.num_sms / (tiles > 0 ? tiles : 1);
  if (ks > nk / 4) ks = nk / 4;
  if (ks > 16) ks = 16;
  const size_t o_bytes = (size_t)T * (L.k + L.S) * L.d * 2;
  while (ks > 1 && ((size_t)ks * T * L.E * sizeof(float) > kRouterPartBytes ||
                    (size_t)ks * T * L.E * sizeof(float) > o_bytes))
    --ks;
  return ks > 1 ? ks : 1;
}

// logits = sum of the K splits' partials, in split order.
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ part, long n, int ksplit,
                                                            float* __restrict__ out) {
  griddep_wait();    // after the predecessor grid (launch.cuh)
  griddep_launch();
  const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float sum = 0.f;
  for (int q = 0; q < ksplit; ++q) sum += part[q * n + i];
  out[i] = sum;
}

cudaError_t launch_tc_router_logits(const Layer& L, const void* x, int T, float* logits, cudaStream_t s,
                                    float* part, size_t part_bytes) {
  CUtensorMap tx, tw;
  if (!make_tmap(&tx, x, L.d, T, BK, BM) || !make_tmap(&tw, L.Wr, L.d, L.E, BK, kBNrouter))
    return cudaErrorInvalidValue;
  TcParams p = {};
  p.dense_rows = T;
  p.K = L.d;
  p.n_tiles = 1;
  p.out = logits;
  p.ldo = L.E;
  p.n_valid = L.E;
  p.status = L.status;
  const int tiles = (T + BM - 1) / BM;
  p.ksplit = tc_router_splits(L, T);
  if (p.ksplit > 1 && (!part || (size_t)p.ksplit * T * L.E * sizeof(float) > part_bytes)) return cudaErrorInvalidValue;
  p.part = part;
  const int total = tiles * p.ksplit;
  cudaError_t e = launch<kBNrouter, A_TMA_K, B_TMA_K, SCHED_DENSE, EPI_F32>(tx, tw, p, total < L.num_sms ? total
                                                                                                    : L.num_sms, s);
  if (e != cudaSuccess || p.ksplit == 1) return e;
  const long n = (long)T * L.E;
  MOE_TRY(launch_pdl(splitk_reduce_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, part, n, p.ksplit,
      logits));
  return cudaGetLastError();
}

TcParams gateup_params(const Layer& L, const Bufs& B, const void* x) {
  TcParams p = base_params(L, B);
  p.A = (const bf16*)x;
  p.lda = L.d;
  p.K = L.d;
  p.n_tiles = 2 * L.f / kBNup;
  p.b_rows_per_seg = 2 * L.f;
  p.out = B.h;
  p.ldo = L.f;
  p.uv = (bf16*)B.uv;
  p.ld_uv = 2 * L.f;
  return p;
}

TcParams down_params(const Layer& L, const Bufs& B) {
  TcParams p = base_params(L, B);
  p.K = L.f;
  p.n_tiles = L.d / kBNdown;
  p.b_rows_per_seg = L.d;
  p.out = B.o;
  p.ldo = L.d;
  p.row_gate = B.row_gate;
  return p;
}

cudaError_t launch_tc_gateup(const Layer& L, const Bufs& B, const void* x, cudaStream_t s) {
  const TcParams p = gateup_params(L, B, x);
  if (use_pairs(L, B))
    return launch<kBNup, A_GATHER_K, B_TMA_K, SCHED_SEG_M, EPI_SWIGLU, 2>(L.tm_W13_h /*unused*/, L.tm_W13_h, p,
                                                                          L.num_sms, s);
  if (use_mt2(L))
    return launch<kBNup, A_GATHER_K, B_TMA_K, SCHED_SEG_M, EPI_SWIGLU, 1, 2>(L.tm_W13 /*unused*/, L.tm_W13, p,
                                                                             L.num_sms, s);
  return launch<kBNup, A_GATHER_K, B_TMA_K, SCHED_SEG_M, EPI_SWIGLU>(L.tm_W13 /*unused*/, L.tm_W13, p, L.num_sms, s);
}

cudaError_t launch_tc_down(const Layer& L, const Bufs& B, cudaStream_t s) {
  CUtensorMap th;
  if (!make_tmap(&th, B.h, L.f, B.R, BK, BM)) return cudaErrorInvalidValue;
  const TcParams p = down_params(L, B);
  if (use_pairs(L, B)) return launch<kBNdown, A_TMA_K, B_TMA_K, SCHED_SEG_M, EPI_GATE, 2>(th, L.tm_Wd_h, p, L.num_sms, s);
  if (use_mt2(L)) return launch<kBNdown, A_TMA_K, B_TMA_K, SCHED_SEG_M, EPI_GATE, 1, 2>(th, L.tm_Wd, p, L.num_sms, s);
  return launch<kBNdown, A_TMA_K, B_TMA_K, SCHED_SEG_M, EPI_GATE>(th, L.tm_Wd, p, L.num_sms, s);
}

// A5 + A6 in one persistent cooperative launch (fused_experts_kernel).
cudaError_t launch_tc_fused_experts(const Layer& L, const Bufs& B, const void* x, cudaStream_t s) {
  static_assert(kBNup == 256 && kBNdown == 256, "the fused kernel runs 128 x 256 tiles");
  CUtensorMap th;
  if (!make_tmap(&th, B.h, L.f, B.R, BK, BM)) return cudaErrorInvalidValue;
  FusedParams q = {};
  q.gu = gateup_params(L, B, x);
  q.dn = down_params(L, B);
  q.dep = L.dep;
  q.done = L.dep_done;
  const int smem = Smem<256, SCHED_SEG_M, 1>::TOTAL;
  static bool attr = false;
  if (!attr) {
    const cudaError_t e = cudaFuncSetAttribute(fused_experts_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;   // every CTA resident: the dependency waits can end
  at[0].val.cooperative = 1;
  cfg.gridDim = dim3(L.num_sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fused_experts_kernel, L.tm_W13, th, L.tm_Wd, q);
}

// The whole forward (routing A1-A4, A5, A6, combine A7) in one cooperative launch
// (fused_forward_kernel). The router splits K exactly as launch_tc_router_logits does, its partials
// in the forward scratch o (which the down tiles write only later).
cudaError_t launch_tc_fused_forward(const Layer& L, const Bufs& B, const void* x, void* y, cudaStream_t s) {
  static_assert(kBNup == 256 && kBNdown == 256 && kBNrouter == 256, "the fused kernels run 128 x 256 tiles");
  if (L.E + L.S > kThreads) return cudaErrorInvalidValue;   // the scan runs on one CTA
  CUtensorMap tx, twr, th;
  if (!make_tmap(&tx, x, L.d, B.T, BK, BM) || !make_tmap(&twr, L.Wr, L.d, L.E, BK, kBNrouter) ||
      !make_tmap(&th, B.h, L.f, B.R, BK, BM))
    return cudaErrorInvalidValue;
  FwdParams q = {};
  TcParams rt = {};
  rt.dense_rows = B.T;
  rt.K = L.d;
  rt.n_tiles = 1;
  rt.out = B.logits;
  rt.ldo = L.E;
  rt.n_valid = L.E;
  rt.status = L.status;
  rt.ksplit = tc_router_splits(L, B.T);
  rt.part = (float*)B.o;
  if (rt.ksplit > 1 && (size_t)rt.ksplit * B.T * L.E * sizeof(float) > (size_t)B.R * L.d * 2)
    return cudaErrorInvalidValue;
  q.rt = rt;
  q.gu = gateup_params(L, B, x);
  q.dn = down_params(L, B);
  q.bias = L.bias;
  q.logits = B.logits;
  q.idx = B.idx;
  q.gate = B.gate;
  q.chunk_hist = B.chunk_hist;
  q.chunk_base = B.chunk_base;
  q.cnt = B.cnt;
  q.off = B.off;
  q.mt_off = B.mt_off;
  q.perm = B.perm;
  q.inv = B.inv;
  q.row_token = B.row_token;
  q.row_gate = B.row_gate;
  q.o = (const bf16*)B.o;
  q.y = (bf16*)y;
  q.T = B.T;
  q.E = L.E;
  q.S = L.S;
  q.k = L.k;
  q.d = L.d;
  q.router = L.router;
  q.renorm = L.renorm;
  q.scale = L.scale;
  q.A = B.A;
  q.nch = B.nch;
  q.dep = L.dep;
  q.dep_len = L.dep_len;
  q.ctr = L.dep_done;
  static bool attr = false;
  if (!attr) {
    const cudaError_t e = cudaFuncSetAttribute(fused_forward_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kFwdSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;   // every CTA resident: the grid barriers and waits can end
  at[0].val.cooperative = 1;
  cfg.gridDim = dim3(L.num_sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kFwdSmem;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fused_forward_kernel, tx, twr, L.tm_W13, th, L.tm_Wd, q);
}

// B1: r = dy_t Wd[e] (K = d; Wd read MN-major), SwiGLU backward, g*h, gate-gradient partials.
cudaError_t launch_tc_bwd_dh(const Layer& L, const Bufs& B, const void* dy, cudaStream_t s) {
  TcParams p = base_params(L, B);
  p.A = (const bf16*)dy;
  p.lda = L.d;
  p.K = L.d;
  p.n_tiles = (L.f + kBNdh - 1) / kBNdh;
  p.b_rows_per_seg = L.d;
  p.out = B.dudv;
  p.out2 = B.hg;
  p.ldo = L.f;
  p.row_gate = B.row_gate;
  p.uv = (bf16*)B.uv;
  p.ld_uv = 2 * L.f;
  p.dg_part = B.dg_part;
  p.dg_slots = L.f / 64;
  if (use_pairs(L, B))
    return launch<kBNdh, A_GATHER_K, B_TMA_MN, SCHED_SEG_M, EPI_DH, 2>(L.tm_Wd_mn /*unused*/, L.tm_Wd_mn, p,
                                                                       L.num_sms, s);
  if (use_mt2(L))
    return launch<kBNdh, A_GATHER_K, B_TMA_MN, SCHED_SEG_M, EPI_DH, 1, 2>(L.tm_Wd_mn /*unused*/, L.tm_Wd_mn, p,
                                                                          L.num_sms, s);
  return launch<kBNdh, A_GATHER_K, B_TMA_MN, SCHED_SEG_M, EPI_DH>(L.tm_Wd_mn /*unused*/, L.tm_Wd_mn, p, L.num_sms,
                                                                  s);
}

// B2: dx_rows = [du dv] W13[e] (K = 2f; W13 read MN-major).
cudaError_t launch_tc_bwd_dx(const Layer& L, const Bufs& B, cudaStream_t s) {
  CUtensorMap ta;
  if (!make_tmap(&ta, B.dudv, 2 * L.f, B.R, BK, BM)) return cudaErrorInvalidValue;
  TcParams p = base_params(L, B);
  p.K = 2 * L.f;
  p.n_tiles = L.d / kBNdx;
  p.b_rows_per_seg = 2 * L.f;
  p.out = B.dx_rows;
  p.ldo = L.d;
  if (use_pairs(L, B)) return launch<kBNdx, A_TMA_K, B_TMA_MN, SCHED_SEG_M, EPI_STORE, 2>(ta, L.tm_W13_mn, p, L.num_sms, s);
  if (use_mt2(L)) return launch<kBNdx, A_TMA_K, B_TMA_MN, SCHED_SEG_M, EPI_STORE, 1, 2>(ta, L.tm_W13_mn, p, L.num_sms, s);
  return launch<kBNdx, A_TMA_K, B_TMA_MN, SCHED_SEG_M, EPI_STORE>(ta, L.tm_W13_mn, p, L.num_sms, s);
}

// B3: dW13[e] = [du dv]_seg^T x_seg, K over the expert's sorted rows.
cudaError_t launch_tc_bwd_dw13(const Layer& L, const Bufs& B, const void* x, void* dWg, void* dWu, bool acc,
                              cudaStream_t s) {
  CUtensorMap tdudv;
  if (!make_tmap(&tdudv, B.dudv, 2 * L.f, B.R, 64, BK)) return cudaErrorInvalidValue;
  TcParams p = base_params(L, B);
  p.Bsrc = (const bf16*)x;
  p.ldb = L.d;
  p.m_tiles = 2 * L.f / BM;
  p.n_tiles = L.d / kBNdw13;
  p.out = dWg;
  p.out2 = dWu;
  p.ldo = L.d;
  p.accumulate = acc ? 1 : 0;
  const uint64_t nseg = L.E + L.S;
  CUtensorMap tg, tu;
  if (!make_tmap(&tg, dWg, L.d, nseg * L.f, 64, 32) || !make_tmap(&tu, dWu, L.d, nseg * L.f, 64, 32))
    return cudaErrorInvalidValue;
  return launch<kBNdw13, A_TMA_MN, B_GATHER_MN, SCHED_SEG_K, EPI_DW13>(tdudv, tdudv /*unused*/, p, L.num_sms, s, &tg,
                                                                       &tu);
}

// B3: dWd[e] = dy_seg^T (g h)_seg, K over the expert's sorted rows: 128 model dimensions (dY rows
// gathered by token, MN-major) by 256 features (g h by TMA) per tile, the dW13 kernel's shape; the
// last feature tile of an odd number of 128-feature blocks runs half empty.
cudaError_t launch_tc_bwd_dwd(const Layer& L, const Bufs& B, const void* dy, void* dWd, bool acc, cudaStream_t s) {
  CUtensorMap thg, td;
  if (!make_tmap(&thg, B.hg, L.f, B.R, 64, BK)) return cudaErrorInvalidValue;
  if (!make_tmap(&td, dWd, L.f, (uint64_t)(L.E + L.S) * L.d, 64, 32)) return cudaErrorInvalidValue;
  TcParams q = base_params(L, B);
  q.A = (const bf16*)dy;
  q.lda = L.d;
  q.m_tiles = L.d / BM;
  q.n_tiles = (L.f + kBNdwd - 1) / kBNdwd;
  q.n_valid = L.f;
  q.out = dWd;
  q.ldo = L.f;
  q.accumulate = acc ? 1 : 0;
  return launch<kBNdwd, A_GATHER_MN, B_TMA_MN, SCHED_SEG_K, EPI_DWD>(thg /*unused*/, thg, q, L.num_sms, s, &td);
}

}  // namespace moe
