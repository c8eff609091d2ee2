// MXFP8 path: E4M3 elements with one E8M0 scale per 32 elements along each
// GEMM's K (OCP Microscaling v1.0), on tcgen05.mma kind::mxf8f6f4 with block
// scales in TMEM.
//
// The MoK page ("Cursor открыл код ядра Mixture of Experts ...", dzen.guru,
// section "Три решения, которые дали результат") names BF16 and MXFP8 support
// for the fused MoE layer. Quantisation here:
//   scale exponent X = floor(log2(amax of the block)) - 8 (E4M3's largest
//   exponent), clamped to [-127, 127], stored as X + 127; elements are
//   round-to-nearest-even E4M3 of v * 2^-X, saturated at +-448.
// Operands per GEMM (all quantised along that GEMM's K):
//   gate/up   x rows (along d)          x  W13 rows (along d)
//   down      h rows (along f)          x  Wd rows (along f)
//   dy.Wd     dy rows (along d)         x  Wd read MN-major, quantised along d
//   dx        [du dv] rows (along 2f)   x  W13 read MN-major, quantised along 2f
//   dW13      [du dv] and x, both along the expert's sorted tokens (32-token
//   dWd       dy and g*h                 blocks, each segment zero-padded to 128;
//                                        chunked step: each chunk's rows at 32)
// Gate/up rows of the MXFP8 W13 are interleaved in blocks of 64 so that one
// 128-column tile holds 64 gate and the matching 64 up features.
//
// The products over token rows gate/up, down and dx run one CTA per 128-row tile and pair of
// 128-column tiles (NB = 2): the staged A tile feeds two MMAs (a 48 KB stage carries 512 MMA cycles)
// and is read from shared memory once per pair. dY.Wd runs one column tile per CTA (NB = 1), whose
// double-buffered accumulators let its heavy epilogue overlap the next tile's MMAs.
// Every operand reaches shared memory through the async proxy, issued by one producer thread per
// stage: TMA tiles for the codes (the token-row activations are quantised in expert-sorted row order,
// so the A tile of a row tile is one rectangular load) and one 512-byte bulk copy per operand for
// the block scales, which every quantiser and epilogue writes in the MMA's atom order (see
// mx_quant.cuh). The MMA thread moves the scales to TMEM with tcgen05.cp.32x128b.warpx4 ahead of the
// stage's MMAs: for a 128-row operand tile the MMA reads row r's four k-block scales (one per 32
// elements of a 128-element stage, selected by the instruction's scale id) from column r/32 of lane
// 32q + (r mod 32) of the lane quadrant q serving the output row, and the warpx4 copy writes the
// atom's 32 x 4 words to all four quadrants. (Per-thread cp.async row gathers and scale loads kept
// the producers issue-bound at ~1,200 cycles per stage, and the MMA thread then needed a proxy
// fence per stage that drained the tensor pipe.)
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"
#include "mx_quant.cuh"
#include "launch.cuh"

namespace moe {

namespace {

constexpr int MBM = 128, MBN = 128, MBK = 128;
constexpr int kProd = 1, kEpi = 4;
constexpr int kMxMmaWarp = kProd + kEpi;
// Warp 0 is the producer (one thread issues every copy), warps 1-4 the epilogue (warp w reads TMEM lane
// quadrant w mod 4), warp 5 issues the scale copies and MMAs, warp 6 tests the ring's full barriers. A test of an mbarrier in the MMA-issuing thread while the tensor pipe runs
// costs a few hundred cycles of idle pipe (the pipe queues only ~1.5 MMAs of work), so that thread never
// tests one: the waiter warp tests each stage's barrier and hands the stage over on a named barrier (one id
// per ring slot), and the epilogue hands back each accumulator on another. Both hand-overs are rendezvous
// (bar.sync on both sides), so no side runs more than one use ahead; after a failed wait a role stops
// waiting but still takes part in every rendezvous, so none is left waiting on a named barrier.
constexpr int kMxWaitWarp = kMxMmaWarp + 1;
constexpr int kMxThreads = (kMxWaitWarp + 1) * 32;
constexpr int kEpiSync = kEpi * 32 + 32;   // a rendezvous of the epilogue warps and the MMA warp
__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// the CTA's share of n units dealt round-robin over the grid
__device__ __forceinline__ int cta_share(int n) {
  return (int)blockIdx.x < n ? (n - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
}
constexpr int kScaleCol0 = 2 * MBN;                                 // TMEM columns after the two accumulators
constexpr int kScaleAtom = 512;   // one 128-row operand's scale words for one K block (32 rows x 16 bytes)
// off[] and the tile prefix mt_off[] (nseg + 1 each), copied to shared memory at kernel start: every
// role maps each unit through them with a shared-memory search.
constexpr int kSegCache = 2 * (kMaxE + 2) * 4;

enum { MB_TMA_K = 0, MB_TMA_MN = 1 };
enum { ME_SWIGLU_Q = 0, ME_GATE = 1, ME_DH_Q = 2, ME_STORE = 3, ME_DW13 = 4, ME_DWD = 5 };

// NB: 128-column B tiles per CTA of the token-row products (1 or 2: with 2, one staged A tile feeds two
// MMAs, so a 48 KB stage carries 512 MMA cycles where a 32 KB one carries 256). Stages, stage bytes,
// the block-scale TMEM columns per stage (A, then each B tile) and the staged scale bytes per stage.
// Shared memory: [scale atoms of every stage][stage ring][barriers][segment cache].
template <int NB> constexpr int mx_stages() { return NB == 2 ? 4 : 6; }
template <int NB> constexpr int mx_stage_bytes() { return MBM * MBK + NB * MBN * MBK; }
template <int NB> constexpr int mx_scale_cols() { return 4 + 4 * NB; }
template <int NB> constexpr int mx_scale_bytes() { return (1 + NB) * kScaleAtom; }
template <int NB> constexpr int mx_scale_region() {
  return (mx_stages<NB>() * mx_scale_bytes<NB>() + 1023) / 1024 * 1024;
}
template <int NB>
constexpr int mx_smem() {
  return mx_scale_region<NB>() + mx_stages<NB>() * mx_stage_bytes<NB>() + 1024 + 256 + kSegCache;
}

struct MxParams {
  const uint8_t* As;      // A scale atoms: by row tile (K-major, atom_tile) or 128-row K group (atom_mn)
  int a_w;                // MN-major A: row width W of the code / scale arrays
  const uint8_t* Bs;      // B scale atoms (K-major weights: atom_k; MN-major: atom_mn)
  int b_w;                // MN-major B: row width W
  int b_rows_per_seg;     // B rows (K-major) or K rows (MN-major) per segment
  const int* row_token;
  const int* off;
  const int* mt_off;
  int nseg;
  int K;                  // token-row products: reduction length (multiple of 128)
  int m_tiles, n_tiles;
  void* out;
  int ldo;
  void* out2;
  uint8_t* oq;            // quantised output codes (ME_SWIGLU_Q: h, ME_DH_Q: dudv)
  uint8_t* os;            // and their scales
  uint8_t *tq, *ts;       // ME_DH_Q: du/dv along the token axis (token-axis operand of dW13), codes and scales
  uint8_t *tq2, *ts2;     // ME_DH_Q: g * h along the token axis (operand of dWd)
  const int* tok_base;    // ME_DH_Q (nullable): row where each segment's token-axis rows start (default mt_off * 128)
  const int* k32;         // weight gradients (nullable): each segment's 32-row K blocks (packed chunk layout)
  const float* row_gate;
  bf16* uv;
  int ld_uv;
  float* dg_part;
  int dg_slots;
  int A_rows;
  int f;
  int accumulate;         // ME_DW13 / ME_DWD: add to the values already in the output
  int* status;
};

// ------------------------------------------------------------- quantise (mx_quant.cuh)
// Scale layouts (all in 512-byte atoms, mx_quant.cuh): the packed weights along K by row (atom_k),
// the expert-sorted activations along K by row tile (atom_tile), the MN-major operands (weights
// quantised along their other axis, token-axis operands) by 128-row K group and column (atom_mn).
enum { SRC_PLAIN = 0, SRC_W13 = 2 };

// Source row of packed W13 row `row` (gate/up interleaved in blocks of G rows).
__device__ __forceinline__ const bf16* w13_src(const bf16* Wg, const bf16* Wu, long row, int f, int G, int K) {
  const long e = row / (2 * f);
  const int pr = (int)(row % (2 * f));
  const int blk = pr / (2 * G), w = pr % (2 * G);
  const int feat = blk * G + (w % G);
  return (w < G ? Wg : Wu) + (e * f + feat) * (long)K;
}

// Along K: one warp per row, one lane per 32-element block.
template <int SRC>
__global__ void __launch_bounds__(256) mx_quant_rows_kernel(const bf16* __restrict__ src, const bf16* __restrict__ src2,
                                                            long rows, int K, int f, int G,
                                                            uint8_t* __restrict__ q, uint8_t* __restrict__ s) {
  const long row = (long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const bf16* sr = SRC == SRC_PLAIN ? src + row * K : w13_src(src, src2, row, f, G, K);
  for (int b = lane; b < K / 32; b += 32) {
    float v[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) unpack8(*reinterpret_cast<const uint4*>(sr + b * 32 + 8 * i), v + 8 * i);
    uint4 lo, hi;
    const uint8_t sc = quant32(v, lo, hi);
    *reinterpret_cast<uint4*>(q + row * K + b * 32) = lo;
    *reinterpret_cast<uint4*>(q + row * K + b * 32 + 16) = hi;
    s[atom_k(row, b, K)] = sc;
  }
}

// Expert-sorted activation rows: CTA per 32-row quarter (blockIdx.y) of a 128-row tile mt of the
// routing's tile prefix (mt_off), one warp per row, one lane per 32-element block. Row r of tile mt of segment e is sorted row
// off[e] + (mt - mt_off[e]) * 128 + r, the token row_token[...] of src (src_rows = T) or, with
// row_token null, that row of src itself; its codes go to q[sorted row] and its scales to the tile's
// atoms. Tile rows past the segment get zero scales (their codes belong to the next segment).
__global__ void __launch_bounds__(256) mx_quant_sorted_kernel(const bf16* __restrict__ src,
                                                              const int* __restrict__ row_token,
                                                              const int* __restrict__ off,
                                                              const int* __restrict__ mt_off, int nseg, int K,
                                                              uint8_t* __restrict__ q, uint8_t* __restrict__ s) {
  griddep_wait();    // after the predecessor grid (launch.cuh)
  griddep_launch();
  __shared__ int seg[3];
  const int mt = blockIdx.x;
  if (threadIdx.x == 0) {
    int lo = -1;
    if (mt < mt_off[nseg]) {
      int l = 0, h = nseg;
      while (h - l > 1) {
        const int mid = (l + h) >> 1;
        if (mt_off[mid] <= mt) l = mid; else h = mid;
      }
      lo = l;
    }
    seg[0] = lo;
    seg[1] = lo >= 0 ? off[lo] + (mt - mt_off[lo]) * 128 : 0;
    seg[2] = lo >= 0 ? off[lo + 1] : 0;
  }
  __syncthreads();
  if (seg[0] < 0) return;
  const int lane = threadIdx.x & 31;
  for (int r = blockIdx.y * 32 + (threadIdx.x >> 5); r < (int)(blockIdx.y + 1) * 32; r += blockDim.x >> 5) {
    const long p = (long)seg[1] + r;
    const bool valid = p < seg[2];
    const bf16* sr = valid ? src + (row_token ? (long)row_token[p] : p) * K : nullptr;
    for (int b = lane; b < K / 32; b += 32) {
      uint8_t sc = 0;
      if (valid) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 4; ++i) unpack8(*reinterpret_cast<const uint4*>(sr + b * 32 + 8 * i), v + 8 * i);
        uint4 lo, hi;
        sc = quant32(v, lo, hi);
        *reinterpret_cast<uint4*>(q + p * K + b * 32) = lo;
        *reinterpret_cast<uint4*>(q + p * K + b * 32 + 16) = hi;
      }
      s[atom_tile(mt, r, b, K)] = sc;
    }
  }
}

enum { CSRC_PLAIN = 0, CSRC_W13 = 1, CSRC_SEG_GATHER = 2 };

// Along rows, in blocks of 32 rows: one warp per 32-row block and 128 columns (4 columns per lane,
// 8-byte loads of each row and one 4-byte store of its codes), 4 warps per CTA. Segment modes write
// each expert's sorted rows at mt_off[e] * 128 (segments padded to 128 rows with zero codes).
template <int SRC>
__global__ void __launch_bounds__(128, 4) mx_quant_cols_kernel(const bf16* __restrict__ src, const bf16* __restrict__ src2,
                                                            const int* __restrict__ row_token,
                                                            const int* __restrict__ off,
                                                            const int* __restrict__ mt_off, int nseg, int W, int f,
                                                            int G, uint8_t* __restrict__ q, uint8_t* __restrict__ s,
                                                            const int* __restrict__ out_base) {
  griddep_wait();    // after the predecessor grid (launch.cuh)
  griddep_launch();
  const int lane = threadIdx.x & 31;
  const int c = (blockIdx.x * 4 + (threadIdx.x >> 5)) * 128 + lane * 4;   // this lane's 4 columns
  long rb = blockIdx.y;                    // 32-row block (of the chunk's padded segment layout)
  if (c >= W) return;                      // W is a multiple of 128: whole warps
  long seg_first = 0, seg_len = 0, seg_src0 = 0, out_shift = 0;
  if (SRC == CSRC_SEG_GATHER) {
    const int pr = (int)(rb * 32);
    if (pr >= mt_off[nseg] * 128) return;
    int lo = 0, hi = nseg;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (mt_off[mid] * 128 <= pr) lo = mid; else hi = mid;
    }
    seg_first = (long)mt_off[lo] * 128;
    seg_len = off[lo + 1] - off[lo];
    seg_src0 = off[lo];
    // out_base (optional): segment lo's rows go to out_base[lo] onwards instead of seg_first, packed at
    // 32 rows: the blocks past the segment's last 32-row block belong to the next chunk's rows there
    if (out_base) {
      if (rb * 32 - seg_first >= ((seg_len + 31) & ~31L)) return;
      out_shift = (long)out_base[lo] - seg_first;
    }
  }
  // source row of row `lane` of the block (null: a zero padding row), then each row's 4 values
  const bf16* my_row = nullptr;
  {
    const long orow = rb * 32 + lane;
    if (SRC == CSRC_PLAIN) my_row = src + orow * W;
    if (SRC == CSRC_W13) my_row = w13_src(src, src2, orow, f, G, W);
    if (SRC == CSRC_SEG_GATHER) {
      const long local = orow - seg_first;
      if (local < seg_len) {
        const long p = seg_src0 + local;
        my_row = src + (long)row_token[p] * W;
      }
    }
  }
  uint2 raw[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const bf16* r = reinterpret_cast<const bf16*>(__shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(my_row), i));
    raw[i] = r ? *reinterpret_cast<const uint2*>(r + c) : make_uint2(0u, 0u);
  }
  // per column: amax over the 32 rows, the block exponent, then the codes (as quant32 does)
  float amax[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    amax[0] = fmaxf(amax[0], fabsf(__uint_as_float(raw[i].x << 16)));
    amax[1] = fmaxf(amax[1], fabsf(__uint_as_float(raw[i].x & 0xffff0000u)));
    amax[2] = fmaxf(amax[2], fabsf(__uint_as_float(raw[i].y << 16)));
    amax[3] = fmaxf(amax[3], fabsf(__uint_as_float(raw[i].y & 0xffff0000u)));
  }
  int X[4];
  float inv[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    X[j] = mx_exponent(amax[j]);
    inv[j] = __uint_as_float((uint32_t)(127 - X[j]) << 23);
  }
  rb += out_shift / 32;                    // segment bases are multiples of 32 rows
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const uint32_t a = __nv_cvt_float2_to_fp8x2(make_float2(__uint_as_float(raw[i].x << 16) * inv[0],
                                                             __uint_as_float(raw[i].x & 0xffff0000u) * inv[1]),
                                                 __NV_SATFINITE, __NV_E4M3);
    const uint32_t b = __nv_cvt_float2_to_fp8x2(make_float2(__uint_as_float(raw[i].y << 16) * inv[2],
                                                             __uint_as_float(raw[i].y & 0xffff0000u) * inv[3]),
                                                 __NV_SATFINITE, __NV_E4M3);
    *reinterpret_cast<uint32_t*>(q + (rb * 32 + i) * W + c) = a | (b << 16);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) s[atom_mn(rb, c + j, W)] = (uint8_t)(X[j] + 127);
}

// Token-axis quantisation inside an epilogue: each lane holds 32 values (columns col0 .. col0 + 31) of
// one row, and the warp's 32 lanes are the 32 consecutive rows of one 32-row block (lanes past the
// segment hold zeros). Column j's block exponent comes from the amax over the lanes (as quant32
// does for one block); the lane's 32 codes go to its row, column col0 + lane's scale to its atom.
__device__ __forceinline__ void quant_tokens32(const float* v, long row, int col0, long W, int lane, uint8_t* q,
                                               uint8_t* s) {
  uint32_t w[8];
  int mine = 0;
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const float a0 = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v[j]))));
    const float a1 = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v[j + 1]))));
    const int X0 = mx_exponent(a0), X1 = mx_exponent(a1);
    const float i0 = __uint_as_float((uint32_t)(127 - X0) << 23), i1 = __uint_as_float((uint32_t)(127 - X1) << 23);
    const uint32_t c = __nv_cvt_float2_to_fp8x2(make_float2(v[j] * i0, v[j + 1] * i1), __NV_SATFINITE, __NV_E4M3);
    if (j & 2) w[j >> 2] |= c << 16;
    else w[j >> 2] = c;
    if (lane == j) mine = X0 + 127;
    if (lane == j + 1) mine = X1 + 127;
  }
  uint4* dst = reinterpret_cast<uint4*>(q + row * W + col0);
  dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
  dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
  s[atom_mn(row >> 5, col0 + lane, W)] = (uint8_t)mine;
}

// ---------------------------------------------------------------- GEMM
__host__ __device__ constexpr uint32_t idesc_mx(int a_mn, int b_mn, int sf_id) {
  return ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) | ((uint32_t)(MBN >> 3) << 17) | (1u << 23) |
         ((uint32_t)(MBM >> 4) << 24) | ((uint32_t)sf_id << 4) | ((uint32_t)sf_id << 29);
}
__device__ __forceinline__ void mma_mx(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                       uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.block32 [%0], "
      "%1, %2, %3, [%4], [%5], p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}
// Shared-memory descriptor of one scale atom for tcgen05.cp: no swizzle, 8-row core matrices of
// 16-byte rows 128 bytes apart (the atom's 32 rows contiguous).
__device__ __forceinline__ uint64_t desc_scale_atom(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)(16 >> 4) << 16) | ((uint64_t)(128 >> 4) << 32) |
         ((uint64_t)1 << 46);
}
// 32 rows x 128 bits from shared memory to TMEM columns taddr .. taddr + 3 of every lane quadrant.
// Ordered before the tcgen05.mma issued after it by the same thread.
__device__ __forceinline__ void tmem_cp_scales(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// Contiguous bytes (16-byte aligned, a multiple of 16) into shared memory, counted on an mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

struct MTile {
  int e, m, n, row0, row_end, nkb;
  int nb;   // B tiles of this unit (n, n+1, ..): 1 or 2
  int mt;   // segment-M: the row tile's index in the tile prefix (its activation scale atoms)
};

// off / mt_off: the shared-memory copies of p.off and p.mt_off
template <int NB>
__device__ __forceinline__ int mx_total(const MxParams& p, const int* mt_off) {
  return mt_off[p.nseg] * ((p.n_tiles + NB - 1) / NB);
}

template <int NB>
__device__ __forceinline__ MTile mx_map(const MxParams& p, int L, const int* off, const int* mt_off) {
  MTile t;
  const int nu = (p.n_tiles + NB - 1) / NB;   // units of NB column tiles
  int lo = 0, hi = p.nseg;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (mt_off[mid] * nu <= L) lo = mid; else hi = mid;
  }
  const int Me = mt_off[lo + 1] - mt_off[lo];
  const int local = L - mt_off[lo] * nu;
  // m-tiles in groups of kRasterM, every column unit of a group before the next group (L2 reuse)
  const int g = local / (kRasterM * nu);
  const int gm = min(kRasterM, Me - g * kRasterM);
  const int within = local - g * kRasterM * nu;
  t.e = lo;
  t.n = NB * (within / gm);
  t.nb = min(NB, p.n_tiles - t.n);
  t.m = g * kRasterM + within % gm;
  t.row0 = off[lo] + t.m * MBM;
  t.row_end = off[lo + 1];
  t.mt = mt_off[lo] + t.m;
  t.nkb = p.K / MBK;
  return t;
}

// Products over the expert-sorted token rows: A = activation rows [R, K] (K-major), B = the expert's
// weight rows (K-major) or columns (MN-major); units of one 128-row tile and NB 128-column tiles.
// NB = 2: the two accumulators fill the TMEM columns that NB = 1 uses for double buffering, so a
// unit's epilogue is not overlapped with the next unit's MMAs.
template <int BMODE, int EPI, int NB>
__global__ void __launch_bounds__(kMxThreads, 1)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, MxParams p) {
  griddep_wait();    // after the predecessor grid (launch.cuh)
  griddep_launch();
  static_assert(mx_smem<NB>() <= 227 * 1024, "shared memory per CTA");
  constexpr int MSTAGES = mx_stages<NB>();
  constexpr int kStageBytes = mx_stage_bytes<NB>();
  constexpr int kScaleBytes = mx_scale_bytes<NB>();
  constexpr int SCOLS = mx_scale_cols<NB>();
  constexpr int NACC = NB == 2 ? 1 : 2;   // accumulator buffers
  constexpr int B_MN = BMODE == MB_TMA_MN ? 1 : 0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* scales = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);   // per stage: A, B (, B2) atoms
  uint8_t* smem = scales + mx_scale_region<NB>();                                    // stage ring (1024-aligned)
  uint64_t* bars = (uint64_t*)(smem + MSTAGES * kStageBytes);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + MSTAGES);
  const uint32_t tfull0 = smem_u32(bars + 2 * MSTAGES);
  const uint32_t drain = smem_u32(bars + 2 * MSTAGES + 4);
  volatile int* abort_flag = (volatile int*)(bars + 2 * MSTAGES + 5);
  uint32_t* tmem_slot = (uint32_t*)(bars + 2 * MSTAGES + 6);
  int* s_off = (int*)(smem_raw + mx_smem<NB>() - kSegCache);   // [kMaxE + 2]
  int* s_mt = s_off + kMaxE + 2;                                       // [kMaxE + 2]
  for (int i = threadIdx.x; i <= p.nseg; i += blockDim.x) {
    s_off[i] = p.off[i];
    s_mt[i] = p.mt_off[i];
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < MSTAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) mbar_init(tfull0 + 8 * a, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMxMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_slot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int ntiles = mx_total<NB>(p, s_mt);
  const int cta_tiles = cta_share(ntiles);
  // named barriers: 1 .. MSTAGES hand over the ring's slots, kAccId + acc the accumulators
  constexpr int kAccId = 1 + MSTAGES;

  if (warp == 0) {
    // ------------------------------------------------------------ producer (one thread)
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int L = blockIdx.x; L < ntiles && ok; L += gridDim.x) {
        const MTile t = mx_map<NB>(p, L, s_off, s_mt);
        for (int kb = 0; kb < t.nkb; ++kb, ++it) {
          const int s = it % MSTAGES;
          const uint32_t ph = (it / MSTAGES) & 1;
          if (!mbar_wait(empty0 + 8 * s, ph ^ 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const uint32_t sa = smem_u32(smem + s * kStageBytes);
          const uint32_t sb = sa + MBM * MBK;
          const uint32_t ssc = smem_u32(scales + s * kScaleBytes);
          const uint32_t fb = full0 + 8 * s;
          const long krowB = (long)t.e * p.b_rows_per_seg + (long)kb * MBK;
          mbar_arrive_expect_tx(fb, (MBM * MBK + kScaleAtom) * (1 + t.nb));
          // codes: A (sorted token rows), the unit's B tiles
          tma_load_2d(sa, &tmA, kb * MBK, t.row0, fb);
          for (int j = 0; j < t.nb; ++j) {   // MBN * MBK bytes apart
            if (BMODE == MB_TMA_K)
              tma_load_2d(sb + j * MBN * MBK, &tmB, kb * MBK, t.e * p.b_rows_per_seg + (t.n + j) * MBN, fb);
            if (BMODE == MB_TMA_MN) tma_load_2d(sb + j * MBN * MBK, &tmB, (t.n + j) * MBN, (int)krowB, fb);
          }
          // block scales: one atom per operand tile
          const long a_atom = (long)t.mt * (p.K / MBK) + kb;
          bulk_load(ssc, p.As + a_atom * kScaleAtom, kScaleAtom, fb);
          for (int j = 0; j < t.nb; ++j) {
            const long b_atom = B_MN ? krowB / MBK * (p.b_w / MBN) + t.n + j
                                     : ((long)t.e * p.b_rows_per_seg / MBN + t.n + j) * (p.K / MBK) + kb;
            bulk_load(ssc + (1 + j) * kScaleAtom, p.Bs + b_atom * kScaleAtom, kScaleAtom, fb);
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == kMxWaitWarp) {
    // ------------------------------------------------ waiter: a stage's operands landed -> the MMA warp
    int it = 0;
    bool dead = false;   // after a failed wait: no more waiting, every rendezvous still made
    for (int L = blockIdx.x; L < ntiles; L += gridDim.x) {
      const MTile t = mx_map<NB>(p, L, s_off, s_mt);
      for (int kb = 0; kb < t.nkb; ++kb, ++it) {
        const int s = it % MSTAGES;
        if (lane == 0 && !dead) dead = !mbar_wait(full0 + 8 * s, (it / MSTAGES) & 1, abort_flag, p.status);
        __syncwarp();
        named_sync(1 + s, 64);
      }
    }
  } else if (warp == kMxMmaWarp) {
    // ----------------------------------------------------------------- MMA (lane 0 issues)
    int it = 0, tcount = 0;
    for (int L = blockIdx.x; L < ntiles; L += gridDim.x, ++tcount) {
      const MTile t = mx_map<NB>(p, L, s_off, s_mt);
      const int acc = tcount % NACC;
      if (tcount >= NACC) named_sync(kAccId + acc, kEpiSync);   // the epilogue has read this accumulator
      const uint32_t dcol = tmem_base + acc * MBN;
      for (int kb = 0; kb < t.nkb; ++kb, ++it) {
        const int s = it % MSTAGES;
        named_sync(1 + s, 64);   // the waiter saw the stage land
        if (lane == 0) {
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * kStageBytes);
          const uint32_t sb = sa + MBM * MBK;
          const uint32_t scol = tmem_base + kScaleCol0 + s * SCOLS;
          const uint32_t ssc = smem_u32(scales + s * kScaleBytes);
          // the stage's scales into TMEM; the previous use of these columns (stage s, MSTAGES K blocks
          // ago) finished before the producers could refill the stage
          tmem_cp_scales(scol, desc_scale_atom(ssc));
          tmem_cp_scales(scol + 4, desc_scale_atom(ssc + kScaleAtom));
          if (NB == 2 && t.nb == 2) tmem_cp_scales(scol + 8, desc_scale_atom(ssc + 2 * kScaleAtom));
          // the stage's first descriptors; the others differ by constants (16-byte units inside the
          // descriptors' 14-bit address field), so little scalar work sits between two MMA issues
          const uint64_t da0 = desc_kmajor(sa), db0 = B_MN ? desc_mnmajor(sb) : desc_kmajor(sb);
          const uint32_t acc0 = kb > 0 ? 1u : 0u;
          const bool two = NB == 2 && t.nb == 2;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t db = db0 + (uint64_t)((B_MN ? k * 4096 : k * 32) >> 4);
            mma_mx(dcol, da0 + (uint64_t)(k * 2), db, idesc_mx(0, B_MN, k), scol, scol + 4, k > 0 ? 1u : acc0);
            if (two)   // the second B tile: its own accumulator, the same A tile
              mma_mx(dcol + MBN, da0 + (uint64_t)(k * 2), db + (uint64_t)((MBN * MBK) >> 4), idesc_mx(0, B_MN, k), scol,
                     scol + 8, k > 0 ? 1u : acc0);
          }
          mma_commit(empty0 + 8 * s);
        }
        __syncwarp();
      }
      if (lane == 0) mma_commit(tfull0 + 8 * acc);
      __syncwarp();
    }
    if (lane == 0) {
      mma_commit(drain);
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
    const int ew = warp & 3;   // TMEM lane quadrant of this warp
    const int r = ew * 32 + lane;
    int tcount = 0;
    bool dead = false;   // after a failed wait: no more waiting or storing, every rendezvous still made
    for (int L = blockIdx.x; L < ntiles; L += gridDim.x, ++tcount) {
      const MTile t0 = mx_map<NB>(p, L, s_off, s_mt);
      const int acc = tcount % NACC;
      if (!dead) dead = !mbar_wait(tfull0 + 8 * acc, (tcount / NACC) & 1, abort_flag, p.status);
      dead = __any_sync(0xffffffffu, dead);   // the warp's lanes take the same path (warp-wide shuffles below)
      tc_fence_after();
      // the unit's column tiles (NB = 2: accumulator jb holds column tile t0.n + jb)
#pragma unroll 1
      for (int jb = 0; jb < (dead ? 0 : t0.nb); ++jb) {
      MTile t = t0;
      t.n = t0.n + jb;
      const uint32_t tbase = tmem_base + (NB == 2 ? jb : acc) * MBN + ((uint32_t)(ew * 32) << 16);
      const int row = t.row0 + r;
      const bool valid = row < t.row_end;
      if (EPI == ME_SWIGLU_Q) {
        // 64 gate (cols 0..63) + 64 up (64..127) accumulators of features n*64..n*64+63
#pragma unroll 1
        for (int c0 = 0; c0 < 64; c0 += 32) {
          uint32_t u[32], v[32];
          tmem_ld32(tbase + c0, u);
          tmem_ld32(tbase + 64 + c0, v);
          tmem_ld_wait();
          if (valid) {
            float hf[32], uf[32], vf[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              uf[i] = __uint_as_float(u[i]);
              vf[i] = __uint_as_float(v[i]);
              hf[i] = silu_f(uf[i]) * vf[i];
            }
            const int col = t.n * 64 + c0;
            uint4 lo, hi;
            const uint8_t sc = quant32(hf, lo, hi);
            *reinterpret_cast<uint4*>(p.oq + (size_t)row * p.f + col) = lo;
            *reinterpret_cast<uint4*>(p.oq + (size_t)row * p.f + col + 16) = hi;
            p.os[atom_tile(t.mt, r, col / 32, p.f)] = sc;
            if (p.uv) {
              bf16* uvrow = p.uv + (size_t)row * p.ld_uv + t.n * 128;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                *reinterpret_cast<uint4*>(uvrow + c0 + q * 8) = pack8(uf + q * 8);
                *reinterpret_cast<uint4*>(uvrow + 64 + c0 + q * 8) = pack8(vf + q * 8);
              }
            }
          }
        }
      } else if (EPI == ME_GATE || EPI == ME_STORE) {
        const float g = (EPI == ME_GATE && valid) ? p.row_gate[row] : 1.f;
        bf16* orow = (bf16*)p.out + (size_t)row * p.ldo + t.n * MBN;
#pragma unroll 1
        for (int c0 = 0; c0 < MBN; c0 += 32) {
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
      } else if (EPI == ME_DH_Q) {
        // r for features n*128 .. n*128+127 = gate/up blocks 2n, 2n+1 (64 features each). du and dv
        // go out quantised along 2f (dx's A operand) and, with g * h, along the token axis (the
        // weight gradients' operands): this warp's 32 rows are one 32-row block of the expert's
        // token-axis rows, which start at tok_base[e] (or mt_off[e] * 128).
        const float g = valid ? p.row_gate[row] : 0.f;
        const long trow = (p.tok_base ? (long)p.tok_base[t.e] : (long)s_mt[t.e] * MBM) + (long)t.m * MBM + r;
        // packed chunk layout (tok_base): a warp block past the segment's last 32-row block is the next chunk's
        const bool tok_block =
            !p.tok_base || t.m * MBM + ew * 32 < ((s_off[t.e + 1] - s_off[t.e] + 31) & ~31);
        float dgp = 0.f;
#pragma unroll 1
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t a[32];
          tmem_ld32(tbase + c0, a);
          tmem_ld_wait();
          const int blk = 2 * t.n + (c0 >> 6), within = c0 & 63;
          const int ucol = blk * 128 + within;          // packed column of u; v at + 64
          float du[32], dv[32], hg[32];
          if (valid) {
            const bf16* urow = p.uv + (size_t)row * p.ld_uv;
            float uf[32], vf[32];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              unpack8(*reinterpret_cast<const uint4*>(urow + ucol + q * 8), uf + q * 8);
              unpack8(*reinterpret_cast<const uint4*>(urow + ucol + 64 + q * 8), vf + q * 8);
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
            uint4 lo, hi;
            uint8_t sc = quant32(du, lo, hi);
            uint8_t* qrow = p.oq + (size_t)row * p.ld_uv;
            *reinterpret_cast<uint4*>(qrow + ucol) = lo;
            *reinterpret_cast<uint4*>(qrow + ucol + 16) = hi;
            p.os[atom_tile(t.mt, r, ucol / 32, 2 * (long)p.f)] = sc;
            sc = quant32(dv, lo, hi);
            *reinterpret_cast<uint4*>(qrow + ucol + 64) = lo;
            *reinterpret_cast<uint4*>(qrow + ucol + 80) = hi;
            p.os[atom_tile(t.mt, r, (ucol + 64) / 32, 2 * (long)p.f)] = sc;
            if ((c0 & 63) == 32) {
              if (row < p.A_rows) p.dg_part[(size_t)row * p.dg_slots + (t.n * 128 + c0 - 32) / 64] = dgp;
              dgp = 0.f;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) du[i] = dv[i] = hg[i] = 0.f;
          }
          if (tok_block) {
            quant_tokens32(du, trow, ucol, 2 * (long)p.f, lane, p.tq, p.ts);
            quant_tokens32(dv, trow, ucol + 64, 2 * (long)p.f, lane, p.tq, p.ts);
            quant_tokens32(hg, trow, t.n * 128 + c0, p.f, lane, p.tq2, p.ts2);
          }
        }
      }
      }   // column tiles of the unit
      tc_fence_before();
      __syncwarp();
      if (tcount + NACC < cta_tiles) named_sync(kAccId + acc, kEpiSync);   // the MMA warp's tile tcount + NACC
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMxMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem_base) : "memory");
  }
}

// One 128 x 128 weight-gradient tile (expert e, row tile m, column tile n) from TMEM to the output,
// by the four epilogue warps (warp ew: rows 32 ew .. 32 ew + 31), each staging its two 32 x 64
// sub-tiles in turn through one 4 KB buffer (128-byte swizzled) and storing each with a TMA operation
// (a 64 x 32 box of the chunked view of the output); the 16 KB this saves over a buffer per sub-tile
// holds a fourth B stage.
// nkb == 0: the expert had no token rows; the tile is zero (or left as it was, accumulating).
template <int EPI>
__device__ __forceinline__ void wgrad_tile_store(const MxParams& p, const CUtensorMap* tmC, const CUtensorMap* tmC2,
                                                 uint32_t wbuf, uint32_t tbase, int e, int m, int n, int nkb, int ew,
                                                 int lane) {
  // Tile rows are packed dW13 rows (blocks of 64 gate then 64 up features: warps 0-1 write dWg rows,
  // warps 2-3 dWu rows) or dWd rows; each warp writes its 32 rows as two 32 x 64 sub-tiles.
  const bool empty = nkb == 0;
  const CUtensorMap* tmo = tmC;
  int orow0;
  if (EPI == ME_DW13) {
    if (ew >= 2) tmo = tmC2;
    orow0 = e * p.f + m * 64 + (ew & 1) * 32;
  } else {
    orow0 = (e * p.m_tiles + m) * MBM + ew * 32;
  }
#pragma unroll 1
  for (int c0 = 0; c0 < MBN; c0 += 64) {
    const uint32_t buf = wbuf;
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
      const bf16* base = (EPI == ME_DW13 && ew >= 2) ? (const bf16*)p.out2 : (const bf16*)p.out;
      const bf16* old = base + (size_t)(orow0 + lane) * p.ldo + n * MBN + c0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float o8[8];
        unpack8(*reinterpret_cast<const uint4*>(old + q * 8), o8);
#pragma unroll
        for (int i = 0; i < 8; ++i) of[q * 8 + i] += o8[i];
      }
    }
    // the warp's previous store must have finished reading the staging
    if (lane == 0) bulk_wait_read<0>();
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
      tma_store_3d_hint(tmo, 0, orow0, n * (MBN / 64) + (c0 >> 6), wbuf, policy_evict_first());
      bulk_commit();
    }
  }
}

// ------------------------------------------------------------------ weight gradients
// dW[e] (rows: the 2f packed gate/up features or d; columns: d or f) = A^T B over the expert's
// sorted token rows; A and B are token-axis operands [Rp, W] (MN-major, 32-row scale blocks; each
// expert's rows start at a multiple of 128 and are zero past its tokens). When an expert's A K groups
// fit in shared memory (at most kWgA * kWgKG of them), a unit is (expert e, 128-row output tile m):
// the CTA keeps them resident and streams the B groups of every column tile n through a ring, so A is
// read once per unit instead of once per output tile; the CTAs of one expert start their column
// sweep at different tiles (row tile m at m * n_tiles / m_tiles), spreading their B requests over the
// expert's tiles. An expert with more K groups streams A with B, and its units are single output
// tiles, dealt round-robin like the rest. A stage holds two 128-row K groups (eight MMAs per B
// stage): the MMA thread's per-stage work (scale copies, commits, the hand-over) leaves the tensor
// pipe idle, since it queues little more than one MMA ahead, and at four MMAs per stage that
// overhead doubled the stage time.
constexpr int kWgKG = 2;            // 128-row K groups per stage (8 MMAs per B stage)
constexpr int kWgA = 2, kWgB = 4;   // resident A stages (up to kWgA * kWgKG K groups), B ring stages
constexpr int kWgStage = kWgKG * MBM * MBK;              // bytes of one operand stage
constexpr int kWgAtoms = kWgKG * kScaleAtom;             // scale bytes of one operand stage
constexpr int kWgOut = kEpi * 32 * 128;                  // epilogue staging: one 32 x 64 bf16 sub-tile per warp
constexpr int kWgScaleRegion = ((kWgA + kWgB) * kWgAtoms + 1023) / 1024 * 1024;
constexpr int kWgSmem = kWgScaleRegion + (kWgA + kWgB) * kWgStage + kWgOut + 1024 + 256 + kSegCache;
static_assert(kWgSmem <= 227 * 1024, "shared memory per CTA");
constexpr int kWgScaleColA = 2 * MBN, kWgScaleColB = kWgScaleColA + 4 * kWgKG * kWgA;   // TMEM scale columns

// Roles as in mx_gemm_kernel; named barriers 1 .. kWgB hand over the B ring's slots (a stage's A, when it
// is loaded, is tested with its B), kWgB + 1 and kWgB + 2 the accumulators.
template <int EPI>
__global__ void __launch_bounds__(kMxThreads, 1)
    mx_wgrad_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmC2, MxParams p) {
  griddep_wait();    // after the predecessor grid (launch.cuh)
  griddep_launch();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* scales = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);   // A stages' atoms, then B's
  uint8_t* sA = scales + kWgScaleRegion;            // kWgA stages (1024-aligned)
  uint8_t* sB = sA + kWgA * kWgStage;               // kWgB stages
  uint8_t* out_stage = sB + kWgB * kWgStage;        // epilogue staging (1024-aligned)
  uint64_t* bars = (uint64_t*)(out_stage + kWgOut);
  const uint32_t afull0 = smem_u32(bars), aempty0 = smem_u32(bars + kWgA);
  const uint32_t bfull0 = smem_u32(bars + 2 * kWgA), bempty0 = smem_u32(bars + 2 * kWgA + kWgB);
  const uint32_t tfull0 = smem_u32(bars + 2 * kWgA + 2 * kWgB);
  const uint32_t drain = tfull0 + 16;
  volatile int* abort_flag = (volatile int*)(bars + 2 * kWgA + 2 * kWgB + 5);
  uint32_t* tmem_slot = (uint32_t*)(bars + 2 * kWgA + 2 * kWgB + 6);
  int* s_mt = (int*)(smem_raw + kWgSmem - kSegCache);   // [kMaxE + 2]: the 128-row block prefix
  int* s_uoff = s_mt + kMaxE + 2;                       // [kMaxE + 2]: the units' prefix over segments
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = p.n_tiles;
  for (int i = threadIdx.x; i <= p.nseg; i += blockDim.x) s_mt[i] = p.mt_off[i];
  if (warp == 0) {
    // units: an A-resident segment has one per row tile (it sweeps every column tile with A held); a
    // streamed segment (A loaded again for every stage anyway) has one per output tile, so its work is
    // dealt over all CTAs instead of landing, one row tile each, on m_tiles of them
    int carry = 0;
    for (int base = 0; base < p.nseg; base += 32) {
      const int e = base + lane;
      int c = 0;
      if (e < p.nseg) {
        const int nst = (p.mt_off[e + 1] - p.mt_off[e] + kWgKG - 1) / kWgKG;
        c = nst <= kWgA ? p.m_tiles : p.m_tiles * nt;
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, c, o);
        if (lane >= o) c += v;
      }
      if (e < p.nseg) s_uoff[e + 1] = carry + c;
      carry += __shfl_sync(0xffffffffu, c, 31);
    }
    if (lane == 0) s_uoff[0] = 0;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kWgA; ++i) {
      mbar_init(afull0 + 8 * i, 1);
      mbar_init(aempty0 + 8 * i, 1);
    }
    for (int i = 0; i < kWgB; ++i) {
      mbar_init(bfull0 + 8 * i, 1);
      mbar_init(bempty0 + 8 * i, 1);
    }
    for (int a = 0; a < 2; ++a) mbar_init(tfull0 + 8 * a, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMxMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_slot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int units = s_uoff[p.nseg];
  // unit u: segment e, row tile m, and its column tiles n0, n0 + 1, ... (mod n_tiles), ntl of them
  struct Unit {
    int e, m, nkb, nst, n0, ntl;
    bool resident;
  };
  auto unit = [&](int u) {
    int lo = 0, hi = p.nseg;   // the segment with s_uoff[e] <= u < s_uoff[e + 1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_uoff[mid] <= u) lo = mid; else hi = mid;
    }
    Unit un;
    un.e = lo;
    un.nkb = s_mt[lo + 1] - s_mt[lo];
    un.nst = (un.nkb + kWgKG - 1) / kWgKG;
    un.resident = un.nst <= kWgA;
    const int local = u - s_uoff[lo];
    if (un.resident) {
      // the row tiles of one expert start their column sweep at different tiles
      un.m = local;
      un.n0 = local * nt / p.m_tiles;
      un.ntl = nt;
    } else {
      un.m = local / nt;
      un.n0 = local % nt;
      un.ntl = 1;
    }
    return un;
  };
  // the column tiles this CTA computes (every role walks the same units, tiles and stages)
  int cta_tiles = 0;
  for (int u = blockIdx.x; u < units; u += gridDim.x) cta_tiles += unit(u).ntl;

  if (warp == 0) {
    // ------------------------------------------------------------ producer (one thread)
    if (lane == 0) {
      int ait = 0, bit = 0;
      bool ok = true;
      // K groups g0 .. g0 + ng - 1 of the stage (tile, 128-row scale atom each) into stage memory dst
      auto load_stage = [&](uint32_t dst, uint32_t sc, const CUtensorMap* tm, const uint8_t* atoms, int w, int col,
                            int row0, int g0, int ng, uint32_t fb) {
        mbar_arrive_expect_tx(fb, ng * (MBM * MBK + kScaleAtom));
        for (int g = 0; g < ng; ++g) {
          const long kg = row0 / MBK + g0 + g;
          tma_load_2d(dst + g * MBM * MBK, tm, col * MBM, row0 + (g0 + g) * MBK, fb);
          bulk_load(sc + g * kScaleAtom, atoms + (kg * (w / MBM) + col) * kScaleAtom, kScaleAtom, fb);
        }
      };
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const Unit un = unit(u);
        const int m = un.m, nkb = un.nkb, nst = un.nst;
        const bool resident = un.resident;
        const int row0 = s_mt[un.e] * MBK;
        for (int i = 0; i < un.ntl && ok; ++i) {
          const int n = (un.n0 + i) % nt;
          for (int st = 0; st < nst; ++st) {
            const int g0 = st * kWgKG, ng = min(kWgKG, nkb - g0);
            if (!resident || i == 0) {
              const int as = ait % kWgA;
              if (!mbar_wait(aempty0 + 8 * as, ((ait / kWgA) & 1) ^ 1, abort_flag, p.status)) {
                ok = false;
                break;
              }
              load_stage(smem_u32(sA + as * kWgStage), smem_u32(scales + as * kWgAtoms), &tmA, p.As, p.a_w, m, row0,
                         g0, ng, afull0 + 8 * as);
              ++ait;
            }
            const int bs = bit % kWgB;
            if (!mbar_wait(bempty0 + 8 * bs, ((bit / kWgB) & 1) ^ 1, abort_flag, p.status)) {
              ok = false;
              break;
            }
            load_stage(smem_u32(sB + bs * kWgStage), smem_u32(scales + (kWgA + bs) * kWgAtoms), &tmB, p.Bs, p.b_w, n,
                       row0, g0, ng, bfull0 + 8 * bs);
            ++bit;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == kMxWaitWarp) {
    // ------------------------------------------------ waiter: a stage's operands landed -> the MMA warp
    int ait = 0, bit = 0;
    bool dead = false;   // after a failed wait: no more waiting, every rendezvous still made
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const Unit un = unit(u);
      const int nst = un.nst;
      const bool resident = un.resident;
      for (int i = 0; i < un.ntl; ++i) {
        for (int st = 0; st < nst; ++st) {
          if (lane == 0 && !dead) {
            if (!resident || i == 0) dead = !mbar_wait(afull0 + 8 * (ait % kWgA), (ait / kWgA) & 1, abort_flag, p.status);
            if (!dead) dead = !mbar_wait(bfull0 + 8 * (bit % kWgB), (bit / kWgB) & 1, abort_flag, p.status);
          }
          if (!resident || i == 0) ++ait;
          __syncwarp();
          named_sync(1 + bit % kWgB, 64);
          ++bit;
        }
      }
    }
  } else if (warp == kMxMmaWarp) {
    // ----------------------------------------------------------------- MMA (lane 0 issues)
    int ait = 0, bit = 0, tcount = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const Unit un = unit(u);
      const int nkb = un.nkb, nst = un.nst;
      const bool resident = un.resident;
      const int k32 = p.k32 ? p.k32[un.e] : 4 * nkb;   // 32-row K blocks that hold rows
      const int ait0 = ait;
      for (int i = 0; i < un.ntl; ++i, ++tcount) {
        const int acc = tcount & 1;
        if (tcount >= 2) named_sync(1 + kWgB + acc, kEpiSync);   // the epilogue has read this accumulator
        const uint32_t dcol = tmem_base + acc * MBN;
        for (int st = 0; st < nst; ++st) {
          const int ng = min(kWgKG, nkb - st * kWgKG);
          const bool load_a = !resident || i == 0;
          const int as = load_a ? ait % kWgA : (ait0 + st) % kWgA;
          const int bs = bit % kWgB;
          named_sync(1 + bs, 64);   // the waiter saw the stage's A (when loaded) and B land
          if (lane == 0) {
            tc_fence_after();
            // the stage's A scales stay in these TMEM columns for every column tile of the unit
            if (load_a)
              for (int g = 0; g < ng; ++g)
                tmem_cp_scales(tmem_base + kWgScaleColA + 4 * (as * kWgKG + g),
                               desc_scale_atom(smem_u32(scales + as * kWgAtoms + g * kScaleAtom)));
            for (int g = 0; g < ng; ++g)
              tmem_cp_scales(tmem_base + kWgScaleColB + 4 * (bs * kWgKG + g),
                             desc_scale_atom(smem_u32(scales + (kWgA + bs) * kWgAtoms + g * kScaleAtom)));
            const uint32_t sa = smem_u32(sA + as * kWgStage), sb = smem_u32(sB + bs * kWgStage);
            for (int g = 0; g < ng; ++g) {
              const int kmax = min(4, k32 - 4 * (st * kWgKG + g));
#pragma unroll
              for (int k = 0; k < 4; ++k)
                if (k < kmax)
                  mma_mx(dcol, desc_mnmajor(sa + g * MBM * MBK + k * 4096),
                         desc_mnmajor(sb + g * MBN * MBK + k * 4096), idesc_mx(1, 1, k),
                         tmem_base + kWgScaleColA + 4 * (as * kWgKG + g), tmem_base + kWgScaleColB + 4 * (bs * kWgKG + g),
                         (st > 0 || g > 0 || k > 0) ? 1u : 0u);
            }
            mma_commit(bempty0 + 8 * bs);
            // an A stage is released after its last use: the unit's last column tile (resident) or this one
            if (!resident || i == un.ntl - 1) mma_commit(aempty0 + 8 * as);
          }
          __syncwarp();
          if (load_a) ++ait;
          ++bit;
        }
        if (lane == 0) mma_commit(tfull0 + 8 * acc);
        __syncwarp();
      }
    }
    if (lane == 0) {
      mma_commit(drain);
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
    const int ew = warp & 3;   // TMEM lane quadrant of this warp
    const uint32_t wbuf = smem_u32(out_stage) + ew * 4096;
    int tcount = 0;
    bool dead = false;   // after a failed wait: no more waiting or storing, every rendezvous still made
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const Unit un = unit(u);
      const int e = un.e, m = un.m, nkb = un.nkb;
      for (int i = 0; i < un.ntl; ++i, ++tcount) {
        const int n = (un.n0 + i) % nt;
        const int acc = tcount & 1;
        if (!dead) dead = !mbar_wait(tfull0 + 8 * acc, (tcount >> 1) & 1, abort_flag, p.status);
        dead = __any_sync(0xffffffffu, dead);   // the warp's lanes take the same path
        if (!dead) {
          tc_fence_after();
          wgrad_tile_store<EPI>(p, &tmC, &tmC2, wbuf, tmem_base + acc * MBN + ((uint32_t)(ew * 32) << 16), e, m, n,
                                nkb, ew, lane);
        }
        tc_fence_before();
        __syncwarp();
        if (tcount + 2 < cta_tiles) named_sync(1 + kWgB + acc, kEpiSync);   // the MMA warp's tile tcount + 2
      }
    }
    // the stores must have read their staging before the CTA exits
    if (lane == 0) bulk_wait<0>();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMxMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem_base) : "memory");
  }
}

template <int EPI>
cudaError_t wg_launch(const CUtensorMap& tmA, const CUtensorMap& tmB, const MxParams& p, int grid, cudaStream_t s,
                      const CUtensorMap& tmC, const CUtensorMap& tmC2) {
  auto kern = mx_wgrad_kernel<EPI>;
  static bool attr = false;
  if (!attr) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kWgSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  MOE_TRY(launch_pdl(kern, dim3(grid), dim3(kMxThreads), kWgSmem, s, tmA, tmB, tmC, tmC2, p));
  return cudaGetLastError();
}

template <int BMODE, int EPI, int NB>
cudaError_t mx_launch(const CUtensorMap& tmA, const CUtensorMap& tmB, const MxParams& p, int grid, cudaStream_t s) {
  auto kern = mx_gemm_kernel<BMODE, EPI, NB>;
  constexpr int smem = mx_smem<NB>();
  static bool attr = false;
  if (!attr) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  MOE_TRY(launch_pdl(kern, dim3(grid), dim3(kMxThreads), smem, s, tmA, tmB, p));
  return cudaGetLastError();
}

MxParams mx_base(const Layer& L, const Bufs& B) {
  MxParams p = {};
  p.row_token = B.row_token;
  p.off = B.off;
  p.mt_off = B.mt_off;
  p.nseg = L.E + L.S;
  p.A_rows = B.A;
  p.f = L.f;
  p.status = L.status;
  return p;
}

inline unsigned blocks_for(long n, int per) { return (unsigned)((n + per - 1) / per); }

}  // namespace

bool mx_supported(const Layer& L) {
  return L.d % 128 == 0 && L.f % 128 == 0 && L.E <= kMaxE && encode_fn() != nullptr;
}

size_t mx_packed_bytes(const Layer& L) {
  const size_t nseg = L.E + L.S, d = L.d, f = L.f;
  auto al = [](size_t v) { return (v + 255) & ~size_t(255); };
  const size_t w13 = nseg * 2 * f * d, wd = nseg * d * f;
  return 2 * (al(w13) + al(w13 / 32)) + 2 * (al(wd) + al(wd / 32));
}

cudaError_t mx_pack_weights(Layer& L, const void* Wg, const void* Wu, const void* Wd, void* base, cudaStream_t s) {
  auto al = [](size_t v) { return (v + 255) & ~size_t(255); };
  const size_t nseg = L.E + L.S, d = L.d, f = L.f;
  const size_t w13 = nseg * 2 * f * d, wd = nseg * d * f;
  uint8_t* p = (uint8_t*)base;
  L.W13q = p; p += al(w13);
  L.W13s = p; p += al(w13 / 32);
  L.W13c = p; p += al(w13);
  L.W13cs = p; p += al(w13 / 32);
  L.Wdq = p; p += al(wd);
  L.Wds = p; p += al(wd / 32);
  L.Wdc = p; p += al(wd);
  L.Wdcs = p; p += al(wd / 32);
  const bf16 *g = (const bf16*)Wg, *u = (const bf16*)Wu, *dw = (const bf16*)Wd;
  const long r13 = (long)nseg * 2 * f, rd = (long)nseg * d;
  mx_quant_rows_kernel<SRC_W13><<<blocks_for(r13, 8), 256, 0, s>>>(g, u, r13, L.d, L.f, kGateMx, L.W13q,
                                                                     L.W13s);
  mx_quant_rows_kernel<SRC_PLAIN><<<blocks_for(rd, 8), 256, 0, s>>>(dw, nullptr, rd, L.f, L.f, 0, L.Wdq,
                                                                     L.Wds);
  MOE_TRY(launch_pdl(mx_quant_cols_kernel<CSRC_W13>, dim3(dim3(blocks_for(d, 512), (unsigned)(r13 / 32))), dim3(128),
      0, s, g, u, nullptr, nullptr, nullptr, 0, L.d, L.f, kGateMx, L.W13c, L.W13cs, nullptr));
  MOE_TRY(launch_pdl(mx_quant_cols_kernel<CSRC_PLAIN>, dim3(dim3(blocks_for(f, 512), (unsigned)(rd / 32))), dim3(128),
      0, s, dw, nullptr, nullptr, nullptr, nullptr, 0, L.f, L.f, 0, L.Wdc, L.Wdcs, nullptr));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (!make_tmap(&L.tm_W13q, L.W13q, d, r13, MBK, MBN, 1) || !make_tmap(&L.tm_Wdq, L.Wdq, f, rd, MBK, MBN, 1) ||
      !make_tmap(&L.tm_W13c, L.W13c, d, r13, MBN, MBK, 1) || !make_tmap(&L.tm_Wdc, L.Wdc, f, rd, MBN, MBK, 1))
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

// Token rows of src [T, K] in expert-sorted order (row_token) with their scale atoms by row tile.
cudaError_t launch_mx_quant_sorted(const Layer& L, const Bufs& B, const void* src, int K, uint8_t* q, uint8_t* s,
                                   cudaStream_t st) {
  const int nseg = L.E + L.S;
  const long tiles = ((long)B.R + 127L * nseg) / 128 + 1;   // at least the routing's tile count
  MOE_TRY(launch_pdl(mx_quant_sorted_kernel, dim3((unsigned)tiles, 4), dim3(256), 0, st, (const bf16*)src, B.row_token,
      B.off, B.mt_off, nseg, K, q, s));
  return cudaGetLastError();
}

// Token rows of src [T, W] (x or dY) along the token axis, the operands of the weight gradients: [Rp, W]
// codes (each segment's rows in sorted order, zero-padded to 128) and atom_mn scales, Rp = mt_off[nseg] * 128.
// out_base (nullable, device [nseg]): row where each segment's rows start in q (default mt_off[e] * 128).
cudaError_t launch_mx_quant_tokens(const Layer& L, const Bufs& B, const void* src, int W, uint8_t* q, uint8_t* s,
                                   cudaStream_t st, const int* out_base) {
  const dim3 grid(blocks_for(W, 512), (unsigned)(B.Rp_max / 32));
  MOE_TRY(launch_pdl(mx_quant_cols_kernel<CSRC_SEG_GATHER>, dim3(grid), dim3(128), 0, st, (const bf16*)src, nullptr,
      B.row_token, B.off, B.mt_off, L.E + L.S, W, 0, 0, q, s, out_base));
  return cudaGetLastError();
}

// Layout of the combined token-axis operands of a chunked step: chunk_off [n][nseg+1] holds each chunk's row
// offsets (off). Expert e's rows of chunk c start at comb_base[c][e]: all chunks of expert e contiguous, in
// chunk order, each padded to a multiple of 32 rows (the token-axis scale block); comb_mt [nseg+1] is the
// prefix of each expert's 128-row groups and comb_k32[e] its 32-row blocks (the weight gradients' MMAs stop
// there; the rest of the last group is never read). One block; thread e per expert (nseg <= 1024).
__global__ void __launch_bounds__(1024) mx_chunk_layout_kernel(const int* __restrict__ chunk_off, int n, int nseg,
                                                                int* __restrict__ comb_base, int* __restrict__ comb_mt,
                                                                int* __restrict__ comb_k32) {
  griddep_wait();    // after the predecessor grid (launch.cuh)
  griddep_launch();
  __shared__ int wsum[32];
  const int e = threadIdx.x, lane = e & 31, w = e >> 5;
  int rows32 = 0;   // this expert's rows over all chunks, each chunk rounded up to 32
  if (e < nseg)
    for (int c = 0; c < n; ++c) rows32 += (chunk_off[c * (nseg + 1) + e + 1] - chunk_off[c * (nseg + 1) + e] + 31) & ~31;
  const int tot = (rows32 + 127) / 128;   // 128-row groups
  int incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[w] = incl;
  __syncthreads();
  int base = 0;
  for (int q = 0; q < w; ++q) base += wsum[q];
  const int excl = base + incl - tot;
  if (e < nseg) {
    comb_mt[e] = excl;
    comb_k32[e] = rows32 / 32;
    int run = excl * 128;
    for (int c = 0; c < n; ++c) {
      comb_base[c * nseg + e] = run;
      run += (chunk_off[c * (nseg + 1) + e + 1] - chunk_off[c * (nseg + 1) + e] + 31) & ~31;
    }
    if (e == nseg - 1) comb_mt[nseg] = excl + tot;
  }
}

cudaError_t launch_mx_chunk_layout(const Layer& L, const int* chunk_off, int n, int* comb_base, int* comb_mt,
                                   int* comb_k32, cudaStream_t st) {
  MOE_TRY(launch_pdl(mx_chunk_layout_kernel, dim3(1), dim3(1024), 0, st, chunk_off, n, L.E + L.S, comb_base, comb_mt,
                     comb_k32));
  return cudaGetLastError();
}

cudaError_t launch_mx_gateup(const Layer& L, const Bufs& B, cudaStream_t s) {
  CUtensorMap ta;
  if (!make_tmap(&ta, B.xq, L.d, B.R, MBK, MBM, 1)) return cudaErrorInvalidValue;
  MxParams p = mx_base(L, B);
  p.As = B.xs;
  p.Bs = L.W13s;
  p.K = L.d;
  p.n_tiles = 2 * L.f / MBN;
  p.b_rows_per_seg = 2 * L.f;
  p.oq = B.hq;
  p.os = B.hs;
  p.uv = (bf16*)B.uv;
  p.ld_uv = 2 * L.f;
  return mx_launch<MB_TMA_K, ME_SWIGLU_Q, 2>(ta, L.tm_W13q, p, L.num_sms, s);
}

cudaError_t launch_mx_down(const Layer& L, const Bufs& B, cudaStream_t s) {
  CUtensorMap th;
  if (!make_tmap(&th, B.hq, L.f, B.R, MBK, MBM, 1)) return cudaErrorInvalidValue;
  MxParams p = mx_base(L, B);
  p.As = B.hs;
  p.Bs = L.Wds;
  p.K = L.f;
  p.n_tiles = L.d / MBN;
  p.b_rows_per_seg = L.d;
  p.out = B.o;
  p.ldo = L.d;
  p.row_gate = B.row_gate;
  return mx_launch<MB_TMA_K, ME_GATE, 2>(th, L.tm_Wdq, p, L.num_sms, s);
}

cudaError_t launch_mx_bwd_dh(const Layer& L, const Bufs& B, const Bufs& O, const int* tok_base, cudaStream_t s) {
  CUtensorMap ta;
  if (!make_tmap(&ta, B.dyq, L.d, B.R, MBK, MBM, 1)) return cudaErrorInvalidValue;
  MxParams p = mx_base(L, B);
  p.As = B.dys;
  p.Bs = L.Wdcs;
  p.b_w = L.f;
  p.K = L.d;
  p.n_tiles = L.f / MBN;
  p.b_rows_per_seg = L.d;
  p.oq = B.dudvq;
  p.os = B.dudvs;
  p.tq = O.dudv_t;
  p.ts = O.dudv_ts;
  p.tq2 = O.hg_t;
  p.ts2 = O.hg_ts;
  p.tok_base = tok_base;
  p.row_gate = B.row_gate;
  p.uv = (bf16*)B.uv;
  p.ld_uv = 2 * L.f;
  p.dg_part = B.dg_part;
  p.dg_slots = L.f / 64;
  // one column tile per CTA: its accumulators double-buffer, so the SwiGLU-backward epilogue of a tile
  // overlaps the next tile's MMAs (measured faster here; the other products keep two column tiles)
  return mx_launch<MB_TMA_MN, ME_DH_Q, 1>(ta, L.tm_Wdc, p, L.num_sms, s);
}

cudaError_t launch_mx_bwd_dx(const Layer& L, const Bufs& B, cudaStream_t s) {
  CUtensorMap ta;
  if (!make_tmap(&ta, B.dudvq, 2 * L.f, B.R, MBK, MBM, 1)) return cudaErrorInvalidValue;
  MxParams p = mx_base(L, B);
  p.As = B.dudvs;
  p.Bs = L.W13cs;
  p.b_w = L.d;
  p.K = 2 * L.f;
  p.n_tiles = L.d / MBN;
  p.b_rows_per_seg = 2 * L.f;
  p.out = B.dx_rows;
  p.ldo = L.d;
  return mx_launch<MB_TMA_MN, ME_STORE, 2>(ta, L.tm_W13c, p, L.num_sms, s);
}

cudaError_t launch_mx_bwd_dw13(const Layer& L, const Bufs& B, void* dWg, void* dWu, bool acc, cudaStream_t s) {
  CUtensorMap ta, tb;
  if (!make_tmap(&ta, B.dudv_t, 2 * L.f, B.Rp_max, MBM, MBK, 1) || !make_tmap(&tb, B.x_t, L.d, B.Rp_max, MBN, MBK, 1))
    return cudaErrorInvalidValue;
  MxParams p = mx_base(L, B);
  p.As = B.dudv_ts;
  p.a_w = 2 * L.f;
  p.Bs = B.x_ts;
  p.b_w = L.d;
  p.m_tiles = 2 * L.f / MBM;
  p.n_tiles = L.d / MBN;
  p.out = dWg;
  p.out2 = dWu;
  p.k32 = B.tok_k32;
  p.ldo = L.d;
  p.accumulate = acc ? 1 : 0;
  const uint64_t nseg = L.E + L.S;
  CUtensorMap tg, tu;
  if (!make_tmap_chunked(&tg, dWg, L.d, nseg * L.f, 32, 1) || !make_tmap_chunked(&tu, dWu, L.d, nseg * L.f, 32, 1))
    return cudaErrorInvalidValue;
  return wg_launch<ME_DW13>(ta, tb, p, L.num_sms, s, tg, tu);
}

cudaError_t launch_mx_bwd_dwd(const Layer& L, const Bufs& B, void* dWd, bool acc, cudaStream_t s) {
  CUtensorMap ta, tb;
  if (!make_tmap(&ta, B.dy_t, L.d, B.Rp_max, MBM, MBK, 1) || !make_tmap(&tb, B.hg_t, L.f, B.Rp_max, MBN, MBK, 1))
    return cudaErrorInvalidValue;
  MxParams p = mx_base(L, B);
  p.As = B.dy_ts;
  p.a_w = L.d;
  p.Bs = B.hg_ts;
  p.b_w = L.f;
  p.m_tiles = L.d / MBM;
  p.n_tiles = L.f / MBN;
  p.out = dWd;
  p.ldo = L.f;
  p.k32 = B.tok_k32;
  p.accumulate = acc ? 1 : 0;
  CUtensorMap td;
  if (!make_tmap_chunked(&td, dWd, L.f, (uint64_t)(L.E + L.S) * L.d, 32, 1)) return cudaErrorInvalidValue;
  return wg_launch<ME_DWD>(ta, tb, p, L.num_sms, s, td, td);
}

}  // namespace moe
