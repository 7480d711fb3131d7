// mx_quant.cu - fused single-pass MX quantiser (BF16 -> E4M3 data + E8M0
// scales) for the row copy (1x32 blocks), the transposed column copy (32x1
// blocks) and the per-group padded column copy.
//
// What is computed follows "DeepSeek-V3 16B FSDP2 MXFP8/HiF8 训练设计" §3 and
// §3.1 (E4M3 data, E8M0 scale, 1x32 / 32x1 blocks, row and col copies), §8.1
// (dynamic quantisation of activations and gradients, dual-axis weights) and
// "低精度训练特性（MXFP8 / HiFloat8）" (block size 32; per-group quantisation
// for the grouped wgrad). Scale rule: X = floor(log2 amax) - 8 clamped to
// [-127, 127], element = E4M3(x * 2**-X) round-to-nearest-even, saturating.
//
// Design: persistent CTAs (several per SM) walk 128x128 tiles of the input.
// In each CTA a producer warp refills a 32 KB shared-memory tile buffer by
// TMA as soon as eight consumer warps have read it, so the next load overlaps
// their conversion and stores; the input is read from HBM exactly once. The
// tile lands as two 64-column halves in the 128-byte swizzled layout (16-byte
// chunk c of row r at c ^ (r % 8)), which makes both passes' shared loads
// bank-conflict free. Row copy: one thread per 1x32 block (a warp covers 8
// rows x 4 blocks), four 16-byte loads, no shuffles, two 16-byte stores.
// Column copy: each thread owns two adjacent columns of one 32-row block.
// amax is an unsigned max over the BF16 magnitude bits (NaN > Inf > finite),
// the exponent comes from its bits, and the conversion is the hardware's
// round-to-nearest-even satfinite E4M3 cvt; blocks holding Inf or NaN take a
// separate path only when some lane of the warp has one.

#include <cuda.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "mx_codec.cuh"
#include "mx_internal.h"
#include "mx_ptx.cuh"

namespace mx {
namespace {

constexpr int kTileRows = 128;
constexpr int kTileCols = 128;
constexpr int kConsumers = 256;               // eight math warps
constexpr int kThreads = kConsumers + 32;     // plus one producer warp
// Tile buffers per CTA. Measured on GB300 (both copies, M x 7168 and
// 8192 x 10944): two buffers per CTA with two CTAs per SM keep the most bytes
// in flight that the shared memory allows next to the column staging buffers
// (+5% over one buffer with three CTAs per SM; fewer CTAs with more rounds
// each, or deeper rings with one CTA per SM, are slower).
#ifndef MX_QUANT_STAGES
#define MX_QUANT_STAGES 2
#endif
constexpr int kStages = MX_QUANT_STAGES;
constexpr int kMaxGroups = MX_MAX_GROUPS;
constexpr int kTileBytes = kTileRows * kTileCols * 2;
constexpr int kHalfCols = 64;  // columns of one swizzled TMA box (128 bytes per row)
// 1: the column copy of a tile goes through a shared-memory staging buffer
// and leaves as whole 128-byte output rows; 0: each thread stores its own
// 32-byte pieces straight to global memory.
#ifndef MX_QUANT_COL_STAGE
#define MX_QUANT_COL_STAGE 1
#endif
constexpr int kColStageBytes = MX_QUANT_COL_STAGE ? kTileCols * kTileRows : 0;  // one E4M3 tile

struct QParams {
  int64_t rows, cols;
  uint8_t* __restrict__ row_data;
  uint8_t* __restrict__ row_scale;
  uint8_t* __restrict__ col_data;
  uint8_t* __restrict__ col_scale;
  const int64_t* __restrict__ offsets;
  int n_groups;
  int64_t col_pitch;
  int64_t row_ka;  // scale-column atoms of the row copy: ceil(cols/128)
  int64_t col_ka;  // scale-column atoms of the column copy: ceil(col_pitch/128)
  int64_t batch;   // stacked matrices (1 unless batched)
  int64_t row_data_bs, row_scale_bs, col_data_bs, col_scale_bs;  // per-matrix output strides, bytes
  int* dev_status;
  uint64_t timeout_ns;
};

// Current scaling (kCur kernels, one matrix or one stack per launch): matrix
// b's scale is amax[b] / fmt in FP32 (1 for an amax that is zero, infinite or
// NaN), written to scale[b]; elements are E4M3(fl32(x / scale)); no scale bytes.
struct CurParams {
  const float* amax;
  float fmt;
  float* scale;
};

// Up to kMaxTensors independent matrices per launch (dense quantisation of
// several operands at once); the grouped and single-matrix calls use one.
constexpr int kMaxTensors = MX_MAX_MULTI;
struct QuantArgs {
  CUtensorMap map[kMaxTensors];
  QParams p[kMaxTensors];
  int64_t tile0[kMaxTensors + 1];  // first launch-wide tile of each tensor; tile0[n] = all tiles
  int n;
};

// The MX block codec (scale rule, element conversion, swizzled scale layout)
// is in mx_codec.cuh, shared with the GEMM epilogue that quantises its output.

// --- current scaling (one FP32 scale per matrix) ---------------------------

// The matrix's scale: amax / format_max as an IEEE FP32 division, or 1 when
// amax is zero, infinite or NaN.
__device__ __forceinline__ float current_scale_of(float amax, float fmt) {
  return (amax > 0.0f && amax <= 3.402823466e38f) ? __fdiv_rn(amax, fmt) : 1.0f;
}

// Division by a matrix's scale s, correctly rounded to FP32. With r = RN(1/s),
// q0 = RN(x * r) lies within one ulp of x / s, the remainder x - q0 * s is
// exact as one FMA, and RN(q0 + (x - q0 * s) * r) is the correctly rounded
// quotient (Markstein's theorem: P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1),
// 1990) while nothing underflows or overflows. q0 = +-0 (x = +-0, or a
// quotient below FP32's normal range) and an infinite q0 are already the
// rounded quotient's value for every E4M3 decision and keep their sign, so
// they are taken as they are. For s >= 2^-100 a subnormal x gives a quotient
// below 2^-26, far below E4M3's smallest subnormal; smaller scales take the
// IEEE division itself (a matrix-uniform branch). Checked against IEEE
// division on every finite BF16 x for every positive finite BF16 amax.
struct CurDiv {
  float s, r;
  bool fast;
};

__device__ __forceinline__ CurDiv cur_div_of(float s) {
  CurDiv d;
  d.s = s;
  d.fast = s >= 7.8886090522101181e-31f;  // 2^-100
  d.r = d.fast ? __frcp_rn(s) : 1.0f;
  return d;
}

__device__ __forceinline__ float cur_div(float x, const CurDiv& d) {
  if (!d.fast) return __fdiv_rn(x, d.s);
  const float q0 = __fmul_rn(x, d.r);
  const float q1 = __fmaf_rn(__fmaf_rn(-q0, d.s, x), d.r, q0);
  return (q0 == 0.0f || fabsf(q0) > 3.402823466e38f) ? q0 : q1;
}

// E4M3 codes of the two BF16 values of w divided by the scale (quotients
// rounded to FP32 first, then to E4M3 nearest-even with saturation); low half
// -> low byte.
__device__ __forceinline__ uint32_t cur_word(uint32_t w, const CurDiv& d) {
  return cvt_pair(cur_div(lo_f(w), d), cur_div(hi_f(w), d));
}

// Replace the code of each NaN half of w by the E4M3 NaN with that half's sign.
__device__ __forceinline__ uint32_t cur_fix_nan(uint32_t c2, uint32_t w) {
  if ((w & 0x7FFFu) > 0x7F80u) c2 = (c2 & 0xFF00u) | 0x7Fu | ((w >> 8) & 0x80u);
  if (((w >> 16) & 0x7FFFu) > 0x7F80u) c2 = (c2 & 0x00FFu) | ((0x7Fu | ((w >> 24) & 0x80u)) << 8);
  return c2;
}

__device__ __forceinline__ bool word_has_nan(uint32_t w) {
  return (w & 0x7FFFu) > 0x7F80u || ((w >> 16) & 0x7FFFu) > 0x7F80u;
}

// Barrier among the eight consumer warps only (the producer warp never joins).
__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

// Exclusive scan of v[0, n) (n <= 4 * blockDim.x) in shared memory; returns
// the total. Every thread of the block must call it.
__device__ int32_t block_exclusive_scan(int32_t* v, int n, int32_t* warp_tot) {
  const int tid = threadIdx.x;
  const int nwarps = blockDim.x >> 5;
  int32_t loc[4];
  int32_t sum = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = tid * 4 + j;
    loc[j] = (i < n) ? v[i] : 0;
    sum += loc[j];
  }
  int32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if ((tid & 31) >= o) incl += t;
  }
  if ((tid & 31) == 31) warp_tot[tid >> 5] = incl;
  __syncthreads();
  int32_t before = 0, total = 0;
  for (int w = 0; w < nwarps; ++w) {
    const int32_t t = warp_tot[w];
    before += (w < (tid >> 5)) ? t : 0;
    total += t;
  }
  int32_t run = before + incl - sum;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = tid * 4 + j;
    if (i < n) v[i] = run;
    run += loc[j];
  }
  __syncthreads();
  return total;
}

struct TileGeo {
  int64_t row0;    // first input row
  int64_t c0;      // first input column
  int64_t kpos;    // first position along the column copy's contraction
  int64_t b;       // stacked matrix
  int valid_rows;  // input rows of this tile that belong to it
  int valid_cols;
};

template <bool kGrouped>
__device__ __forceinline__ TileGeo tile_geo(const QParams& p, int64_t t, int64_t col_tiles, int64_t row_tiles,
                                            const int32_t* g_off, const int32_t* g_tile) {
  TileGeo g;
  g.b = t / (row_tiles * col_tiles);
  t -= g.b * row_tiles * col_tiles;
  const int64_t rt = t / col_tiles;
  const int64_t ct = t - rt * col_tiles;
  g.c0 = ct * kTileCols;
  g.valid_cols = static_cast<int>(min64(kTileCols, p.cols - g.c0));
  if constexpr (kGrouped) {
    const int32_t tp = static_cast<int32_t>(rt);
    int lo = 0, hi = p.n_groups - 1;  // last group e with g_tile[e] <= tp (it is non-empty)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (g_tile[mid] <= tp) lo = mid; else hi = mid - 1;
    }
    const int lt = tp - g_tile[lo];
    g.row0 = static_cast<int64_t>(g_off[lo]) + static_cast<int64_t>(lt) * kTileRows;
    g.valid_rows = min(kTileRows, g_off[lo + 1] - g_off[lo] - lt * kTileRows);
    g.kpos = rt * kTileRows;
  } else {
    g.row0 = rt * kTileRows;
    g.valid_rows = static_cast<int>(min64(kTileRows, p.rows - g.row0));
    g.kpos = g.row0;
  }
  return g;
}

// Bounded wait that also gives up once another thread of the CTA has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, const QParams& p,
                                              volatile int32_t* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > p.timeout_ns) {
      *abort_flag = 1;
      if (p.dev_status) atomicExch(p.dev_status, static_cast<int>(MX_ERR_TIMEOUT));
      return false;
    }
  }
}

// Two resident CTAs per SM.
#ifndef MX_QUANT_MIN_BLOCKS
#define MX_QUANT_MIN_BLOCKS 2
#endif

// kMulti: the launch holds several matrices and each tile looks up its own;
// otherwise every tile belongs to matrix 0 and its fields stay fixed
// parameter operands.
// The body of both quantiser kernels below: block scales (MX) or one
// current scale per matrix (kCur).
template <bool kRow, bool kCol, bool kGrouped, bool kMulti, bool kCur>
__device__ __forceinline__ void quant_body(const QuantArgs& qa, const CurParams& cur) {
  static_assert(!kCur || !kMulti, "current scaling: one matrix (or one stack) per launch");
  const QParams& p = qa.p[0];  // grouped and shared fields (status word, bound)
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment: the unit of the 128-byte swizzle pattern.
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tiles = smem;  // kStages x 2 halves x [128 rows][128 bytes], swizzled
  uint8_t* col_stage = smem + kStages * kTileBytes;                  // 2 x [128 out rows][128 bytes], swizzled
  uint8_t* col_sc = col_stage + 2 * kColStageBytes;                  // 2 x [128][4] column-copy scales
  uint64_t* full = reinterpret_cast<uint64_t*>(col_sc + 1024);       // [kStages] tile landed
  uint64_t* empty = full + kStages;                                  // [kStages] tile consumed
  int32_t* g_off = reinterpret_cast<int32_t*>(empty + kStages);      // [E+1] row offsets
  int32_t* g_tile = g_off + (kMaxGroups + 1);                        // [E+1] padded tile starts
  __shared__ int32_t warp_tot[kThreads / 32];
  __shared__ int32_t s_bad;
  __shared__ int32_t s_total_tiles;
  __shared__ volatile int32_t s_abort;
  // Each stage's tile geometry (and tensor, several tensors per launch), written
  // by the producer before its arrival on the stage's full barrier.
  __shared__ TileGeo s_geo[kStages];
  __shared__ int32_t s_geo_ti[kStages];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // What touches no global memory runs before the wait for the previous
  // kernel: the stage barriers and the tensor-map prefetch (the maps are
  // kernel parameters).
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == kConsumers / 32 && lane == 0)
    for (int i = 0; i < qa.n; ++i) tma_prefetch_desc(&qa.map[i]);
  // Programmatic dependent launch: let the next kernel on the stream be
  // scheduled, and touch global memory only once the previous one completed.
  pdl_launch_dependents();
  pdl_wait();

  const int64_t col_tiles = (p.cols + kTileCols - 1) / kTileCols;
  int64_t row_tiles = (p.rows + kTileRows - 1) / kTileRows;

  if constexpr (kGrouped) {
    const int E = p.n_groups;
    if (tid == 0) s_bad = 0;
    __syncthreads();
    for (int e = tid; e <= E; e += kThreads) {
      const int64_t o = p.offsets[e];
      g_off[e] = static_cast<int32_t>(o);
      bool bad = (o < 0) || (o > p.rows) || (e == 0 && o != 0) || (e == E && o != p.rows);
      if (e > 0 && o < p.offsets[e - 1]) bad = true;
      if (bad) s_bad = 1;
    }
    __syncthreads();
    if (s_bad == 0) {
      for (int e = tid; e < E; e += kThreads) g_tile[e] = (g_off[e + 1] - g_off[e] + kTileRows - 1) / kTileRows;
      __syncthreads();
      const int32_t total = block_exclusive_scan(g_tile, E, warp_tot);
      if (tid == 0) {
        g_tile[E] = total;
        s_total_tiles = total;
        if (static_cast<int64_t>(total) * kTileRows > p.col_pitch) s_bad = 1;
      }
    }
    __syncthreads();
    if (s_bad) {
      if (tid == 0 && blockIdx.x == 0 && p.dev_status) atomicExch(p.dev_status, static_cast<int>(MX_ERR_DEVICE_CHECK));
      return;
    }
    row_tiles = s_total_tiles;
    // Row-scale padding rows [rows, ceil(rows/128)*128) belong to no group tile.
    if (kRow && !kCur) {
      const int64_t padded = (p.rows + kTileRows - 1) / kTileRows * kTileRows;
      for (int64_t ct = blockIdx.x; ct < col_tiles; ct += gridDim.x)
        for (int64_t r = p.rows + tid; r < padded; r += kThreads)
          *reinterpret_cast<uint32_t*>(p.row_scale + scale_offset(r, ct * (kTileCols / 32), p.row_ka)) = 0u;
    }
  }

  // Grouped launches hold one matrix and take their tile grid from the groups.
  const int64_t ntiles = kGrouped ? row_tiles * col_tiles : qa.tile0[qa.n];
  if constexpr (kCur) {
    // the scale each matrix was quantised with, for the GEMM that reads it
    if (blockIdx.x == 0)
      for (int64_t b = tid; b < p.batch; b += kThreads) cur.scale[b] = current_scale_of(cur.amax[b], cur.fmt);
  }
  __syncthreads();

  if (warp == kConsumers / 32) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int j = 0;
      int ti = 0;  // tensor of tile t (t only grows)
      int last_phase_issued[kStages];
#pragma unroll
      for (int s = 0; s < kStages; ++s) last_phase_issued[s] = -1;
      for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++j) {
        const int s = j % kStages;
        const uint32_t ph = static_cast<uint32_t>((j / kStages) & 1);
        if (!wait_or_abort(&empty[s], ph ^ 1u, p, &s_abort)) break;
        if constexpr (kMulti)
          while (t >= qa.tile0[ti + 1]) ++ti;
        const QParams& pt = qa.p[ti];
        const TileGeo g =
            kGrouped ? tile_geo<kGrouped>(p, t, col_tiles, row_tiles, g_off, g_tile)
                     : tile_geo<kGrouped>(pt, t - qa.tile0[ti], (pt.cols + kTileCols - 1) / kTileCols,
                                          (pt.rows + kTileRows - 1) / kTileRows, g_off, g_tile);
        s_geo[s] = g;
        s_geo_ti[s] = ti;
        mbar_arrive_expect_tx(&full[s], kTileBytes);  // releases the two words above with the stage
#pragma unroll
        for (int h = 0; h < 2; ++h)
          tma_load_3d(tiles + s * kTileBytes + h * (kTileBytes / 2), &qa.map[ti], &full[s],
                      static_cast<int32_t>(g.c0 + h * kHalfCols), static_cast<int32_t>(g.row0),
                      static_cast<int32_t>(g.b));
#pragma unroll
        for (int q = 0; q < kStages; ++q)
          if (q == s) last_phase_issued[q] = static_cast<int>(ph);
      }
      if (s_abort) {
        // Let the loads this CTA issued land before it leaves.
#pragma unroll
        for (int q = 0; q < kStages; ++q)
          if (last_phase_issued[q] >= 0) mbar_wait(&full[q], static_cast<uint32_t>(last_phase_issued[q]), p.timeout_ns);
      }
    }
  } else {
    // ----------------------------------------------------------- consumers
    int j = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++j) {
      const int s = j % kStages;
      const uint32_t ph = static_cast<uint32_t>((j / kStages) & 1);
      // Every consumer runs every iteration (and every consumers_sync) even
      // after an abort, so the named barrier can never strand a warp.
      const bool ok = !s_abort && wait_or_abort(&full[s], ph, qa.p[0], &s_abort);
      // The tile's geometry and tensor as the producer published them with
      // the stage; read before this thread releases the stage.
      TileGeo g{};
      int ti = 0;
      if (ok) {
        g = s_geo[s];
        if constexpr (kMulti) ti = s_geo_ti[s];
      }
      const QParams& p = qa.p[ti];
      uint8_t* const row_data = p.row_data + g.b * p.row_data_bs;
      uint8_t* const row_scale = p.row_scale + g.b * p.row_scale_bs;
      uint8_t* const col_data = p.col_data + g.b * p.col_data_bs;
      uint8_t* const col_scale = p.col_scale + g.b * p.col_scale_bs;
      const uint32_t* tile = reinterpret_cast<const uint32_t*>(tiles + s * kTileBytes);
      const uint4* tile16 = reinterpret_cast<const uint4*>(tiles + s * kTileBytes);
      uint8_t* csc = col_sc + (j & 1) * 512;
      CurDiv cs{1.0f, 1.0f, true};  // current scaling: this tile's matrix scale
      if constexpr (kCur) cs = cur_div_of(current_scale_of(__ldg(cur.amax + g.b), cur.fmt));

      if (kRow && ok) {
        // ---- row copy: one thread per 1x32 block; lanes 8b..8b+7 take block b
        // of eight consecutive rows, so each 8-lane load phase reads eight
        // distinct swizzled chunk positions.
        const int blk = lane >> 3;
        const int rsub = lane & 7;
        const uint4* src = tile16 + (blk >> 1) * (kTileRows * 8) + rsub * 8;
        const int cbase = (blk & 1) * 4;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int r0 = i * 64 + warp * 8;
          const int r = r0 + rsub;
          uint4 v[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) v[j] = src[r0 * 8 + ((cbase + j) ^ rsub)];
          if constexpr (kCur) {
            const int64_t grow = g.row0 + r;
            uint32_t q[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              q[2 * j] = cur_word(v[j].x, cs) | (cur_word(v[j].y, cs) << 16);
              q[2 * j + 1] = cur_word(v[j].z, cs) | (cur_word(v[j].w, cs) << 16);
            }
            bool has_nan = false;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              has_nan |= word_has_nan(v[j].x) | word_has_nan(v[j].y) | word_has_nan(v[j].z) | word_has_nan(v[j].w);
            if (__any_sync(0xFFFFFFFFu, has_nan) && has_nan) {
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                q[2 * j] = cur_fix_nan(q[2 * j] & 0xFFFFu, v[j].x) | (cur_fix_nan(q[2 * j] >> 16, v[j].y) << 16);
                q[2 * j + 1] =
                    cur_fix_nan(q[2 * j + 1] & 0xFFFFu, v[j].z) | (cur_fix_nan(q[2 * j + 1] >> 16, v[j].w) << 16);
              }
            }
            if (r < g.valid_rows && blk * 32 < g.valid_cols) {
              uint4* dst = reinterpret_cast<uint4*>(row_data + grow * p.cols + g.c0 + blk * 32);
              dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
              dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
            }
            if constexpr (kCol) {
              // One scale for the whole matrix: the column copy holds the same
              // codes, transposed. They replace the first two of the four
              // 16-byte chunks this thread read (its own), for the column pass.
              uint4* own = const_cast<uint4*>(src) + r0 * 8;
              own[cbase ^ rsub] = make_uint4(q[0], q[1], q[2], q[3]);
              own[(cbase + 1) ^ rsub] = make_uint4(q[4], q[5], q[6], q[7]);
            }
            continue;
          }
          uint32_t m = 0;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            m = __vmaxu2(__vmaxu2(m, __vmaxu2(v[j].x & 0x7FFF7FFFu, v[j].y & 0x7FFF7FFFu)),
                         __vmaxu2(v[j].z & 0x7FFF7FFFu, v[j].w & 0x7FFF7FFFu));
          const uint32_t code = scale_code(half_max(m));
          const bool nan_block = (code == 0xFFu);
          const float inv = inv_scale(nan_block ? 0u : code);
          uint32_t q[8];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            q[2 * j] = quant_quad(v[j].x, v[j].y, inv);
            q[2 * j + 1] = quant_quad(v[j].z, v[j].w, inv);
          }
          if (__any_sync(0xFFFFFFFFu, nan_block) && nan_block) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              q[2 * j] = nan_pair(v[j].x) | (nan_pair(v[j].y) << 16);
              q[2 * j + 1] = nan_pair(v[j].z) | (nan_pair(v[j].w) << 16);
            }
          }
          const int64_t grow = g.row0 + r;
          if (r < g.valid_rows && blk * 32 < g.valid_cols) {
            uint4* dst = reinterpret_cast<uint4*>(row_data + grow * p.cols + g.c0 + blk * 32);
            dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
            dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
          }
          // Dense: rows past the end (zero-filled by the TMA) write the zero
          // codes of the scale padding. Grouped: those rows belong to the next
          // group's tile.
          const bool write_scale = kGrouped ? (r < g.valid_rows) : true;
          if (write_scale) row_scale[scale_offset(grow, (g.c0 >> 5) + blk, p.row_ka)] = static_cast<uint8_t>(code);
        }
      }

      if constexpr (kCol) {
        if constexpr (kCur && kRow) {
          // Current scaling with both copies: the row pass left every code in
          // the tile (the 32 codes of row r, columns 32b .. 32b + 31, in
          // 16-byte chunks 4(b % 2) and 4(b % 2) + 1 of row r of half b / 2,
          // swizzled like the input). Once all of them are there, the column
          // copy only transposes bytes.
          consumers_sync();
          if (ok) {
            const int cp = tid & 63;
            const int rb = tid >> 6;
            const uint8_t* half = tiles + s * kTileBytes + (cp >> 5) * (kTileBytes / 2);
            const int chunk = ((cp >> 4) & 1) * 4 + ((cp >> 3) & 1);
            const int byte = 2 * (cp & 7);
            uint8_t* stg = col_stage + (j & 1) * kColStageBytes;
            // rows 16u .. 16u + 15 of the block: one 16-byte output chunk per column
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              uint32_t c[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int r = rb * 32 + 16 * u + i;
                c[i] = *reinterpret_cast<const uint16_t*>(half + r * 128 + ((chunk ^ (r & 7)) << 4) + byte);
              }
              if (u == 1) mbar_arrive(&empty[s]);  // this thread is done with the tile
              if (kGrouped && g.valid_rows < kTileRows) {
                // rows past the group's end hold the next group's data: zero padding
#pragma unroll
                for (int i = 0; i < 16; ++i)
                  if (rb * 32 + 16 * u + i >= g.valid_rows) c[i] = 0u;
              }
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                uint32_t o[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  // byte h of rows 4q .. 4q + 3
                  const uint32_t t01 = __byte_perm(c[4 * q], c[4 * q + 1], 0x5140);
                  const uint32_t t23 = __byte_perm(c[4 * q + 2], c[4 * q + 3], 0x5140);
                  o[q] = __byte_perm(t01, t23, h ? 0x7632 : 0x5410);
                }
                const int orow = 2 * cp + h;
                *reinterpret_cast<uint4*>(stg + orow * 128 + (((2 * rb + u) ^ (orow & 7)) << 4)) =
                    make_uint4(o[0], o[1], o[2], o[3]);
              }
            }
          }
        } else if (ok) {
          // ---- column copy: thread = (column pair cp, 32-row block rb) ----
          const int cp = tid & 63;
          const int rb = tid >> 6;
          // Word cp of a 256-byte row: half cp / 32, chunk (cp / 4) % 8, word cp % 4.
          const uint32_t* src = tile + (cp >> 5) * (kTileRows * 32) + rb * 32 * 32 + (cp & 3);
          const int cc = (cp >> 2) & 7;
          uint32_t w[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) w[i] = src[i * 32 + ((cc ^ (i & 7)) << 2)];
          mbar_arrive(&empty[s]);  // this thread is done with the tile
          if (kGrouped && g.valid_rows < kTileRows) {
            // rows past the group's end hold the next group's data: they count as zero padding
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (rb * 32 + i >= g.valid_rows) w[i] = 0u;
          }
          if constexpr (kCur) {
            // One column at a time, straight into the staging tile (fewer live
            // registers beside the division's).
            static_assert(MX_QUANT_COL_STAGE, "current scaling stages its column copy");
            bool has_nan = false;
#pragma unroll
            for (int i = 0; i < 32; ++i) has_nan |= word_has_nan(w[i]);
            const bool fix = __any_sync(0xFFFFFFFFu, has_nan) && has_nan;
            uint8_t* stg = col_stage + (j & 1) * kColStageBytes;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t o[8];
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const uint32_t a = w[4 * q], bb = w[4 * q + 1], c = w[4 * q + 2], d = w[4 * q + 3];
                const float fa = h ? hi_f(a) : lo_f(a), fb = h ? hi_f(bb) : lo_f(bb);
                const float fc = h ? hi_f(c) : lo_f(c), fd = h ? hi_f(d) : lo_f(d);
                o[q] = cvt_pair(cur_div(fa, cs), cur_div(fb, cs)) | (cvt_pair(cur_div(fc, cs), cur_div(fd, cs)) << 16);
                if (fix) {
                  // the halves of column 2cp + h, rows 4q .. 4q + 3
                  const uint32_t ab = h ? ((a >> 16) | (bb & 0xFFFF0000u)) : ((a & 0xFFFFu) | (bb << 16));
                  const uint32_t cd = h ? ((c >> 16) | (d & 0xFFFF0000u)) : ((c & 0xFFFFu) | (d << 16));
                  o[q] = cur_fix_nan(o[q] & 0xFFFFu, ab) | (cur_fix_nan(o[q] >> 16, cd) << 16);
                }
              }
              // output row 2cp + h, 16-byte chunks 2rb and 2rb + 1; chunk q of row o at q ^ (o % 8)
              const int orow = 2 * cp + h;
              *reinterpret_cast<uint4*>(stg + orow * 128 + (((2 * rb) ^ (orow & 7)) << 4)) =
                  make_uint4(o[0], o[1], o[2], o[3]);
              *reinterpret_cast<uint4*>(stg + orow * 128 + (((2 * rb + 1) ^ (orow & 7)) << 4)) =
                  make_uint4(o[4], o[5], o[6], o[7]);
            }
          } else {
            uint32_t m = 0;
#pragma unroll
            for (int i = 0; i < 32; ++i) m = __vmaxu2(m, w[i] & 0x7FFF7FFFu);
            const uint32_t code_lo = scale_code(m & 0xFFFFu);
            const uint32_t code_hi = scale_code(m >> 16);
            const bool nan_lo = code_lo == 0xFFu, nan_hi = code_hi == 0xFFu;
            const float inv_lo = inv_scale(nan_lo ? 0u : code_lo);
            const float inv_hi = inv_scale(nan_hi ? 0u : code_hi);
            uint32_t out_lo[8], out_hi[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const uint32_t a = w[4 * q], bb = w[4 * q + 1], c = w[4 * q + 2], d = w[4 * q + 3];
              out_lo[q] = cvt_pair(lo_f(a) * inv_lo, lo_f(bb) * inv_lo) |
                          (cvt_pair(lo_f(c) * inv_lo, lo_f(d) * inv_lo) << 16);
              out_hi[q] = cvt_pair(hi_f(a) * inv_hi, hi_f(bb) * inv_hi) |
                          (cvt_pair(hi_f(c) * inv_hi, hi_f(d) * inv_hi) << 16);
            }
            if (__any_sync(0xFFFFFFFFu, nan_lo || nan_hi)) {
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const uint32_t a = w[4 * q], bb = w[4 * q + 1], c = w[4 * q + 2], d = w[4 * q + 3];
                if (nan_lo)
                  out_lo[q] = nan_pair((a & 0xFFFFu) | (bb << 16)) | (nan_pair((c & 0xFFFFu) | (d << 16)) << 16);
                if (nan_hi)
                  out_hi[q] = nan_pair((a >> 16) | (bb & 0xFFFF0000u)) | (nan_pair((c >> 16) | (d & 0xFFFF0000u)) << 16);
              }
            }
            csc[(2 * cp) * 4 + rb] = static_cast<uint8_t>(code_lo);
            csc[(2 * cp + 1) * 4 + rb] = static_cast<uint8_t>(code_hi);
#if MX_QUANT_COL_STAGE
          // Output rows 2cp and 2cp+1, 16-byte chunks 2rb and 2rb+1 of the
          // tile's 128 bytes along K; chunk q of row o sits at q ^ (o % 8).
          uint8_t* stg = col_stage + (j & 1) * kColStageBytes;
          const int o0 = 2 * cp, o1 = 2 * cp + 1;
          *reinterpret_cast<uint4*>(stg + o0 * 128 + (((2 * rb) ^ (o0 & 7)) << 4)) =
              make_uint4(out_lo[0], out_lo[1], out_lo[2], out_lo[3]);
          *reinterpret_cast<uint4*>(stg + o0 * 128 + (((2 * rb + 1) ^ (o0 & 7)) << 4)) =
              make_uint4(out_lo[4], out_lo[5], out_lo[6], out_lo[7]);
          *reinterpret_cast<uint4*>(stg + o1 * 128 + (((2 * rb) ^ (o1 & 7)) << 4)) =
              make_uint4(out_hi[0], out_hi[1], out_hi[2], out_hi[3]);
          *reinterpret_cast<uint4*>(stg + o1 * 128 + (((2 * rb + 1) ^ (o1 & 7)) << 4)) =
              make_uint4(out_hi[4], out_hi[5], out_hi[6], out_hi[7]);
#else
          const int64_t c = g.c0 + 2 * cp;
          const bool block_valid = kGrouped ? true : (rb * 32 < g.valid_rows);
          if (block_valid) {
            const int64_t k = g.kpos + rb * 32;
            if (c < p.cols) {
              uint4* dst = reinterpret_cast<uint4*>(col_data + c * p.col_pitch + k);
              dst[0] = make_uint4(out_lo[0], out_lo[1], out_lo[2], out_lo[3]);
              dst[1] = make_uint4(out_lo[4], out_lo[5], out_lo[6], out_lo[7]);
            }
            if (c + 1 < p.cols) {
              uint4* dst = reinterpret_cast<uint4*>(col_data + (c + 1) * p.col_pitch + k);
              dst[0] = make_uint4(out_hi[0], out_hi[1], out_hi[2], out_hi[3]);
              dst[1] = make_uint4(out_hi[4], out_hi[5], out_hi[6], out_hi[7]);
            }
          }
#endif
          }  // block scales
        }
        // The four 32-row blocks of a column sit in four warps: gather their
        // scale bytes (double-buffered by iteration, so one barrier suffices).
        consumers_sync();
#if MX_QUANT_COL_STAGE
        if (ok) {
          // Whole output rows: eight lanes per 128-byte row, 16 bytes each.
          const uint8_t* stg = col_stage + (j & 1) * kColStageBytes;
#pragma unroll
          for (int it = 0; it < (kTileCols * 8) / kConsumers; ++it) {
            const int idx = it * kConsumers + tid;
            const int o = idx >> 3;
            const int q = idx & 7;
            const int64_t c = g.c0 + o;
            // Dense: rows past the end of the input form no block. Grouped:
            // a segment's padding rows are zeros that must be written.
            const bool chunk_valid = kGrouped ? true : (q * 16 < g.valid_rows);
            if (c < p.cols && chunk_valid)
              *reinterpret_cast<uint4*>(col_data + c * p.col_pitch + g.kpos + q * 16) =
                  *reinterpret_cast<const uint4*>(stg + o * 128 + ((q ^ (o & 7)) << 4));
          }
        }
#endif
        if (!kCur && ok && tid < kTileCols) {
          const uint32_t word = *reinterpret_cast<const uint32_t*>(csc + tid * 4);
          *reinterpret_cast<uint32_t*>(col_scale + scale_offset(g.c0 + tid, g.kpos >> 5, p.col_ka)) = word;
        }
      } else {
        if (ok) mbar_arrive(&empty[s]);
      }
    }
  }
}

template <bool kRow, bool kCol, bool kGrouped, bool kMulti>
__global__ void __launch_bounds__(kThreads, MX_QUANT_MIN_BLOCKS)
    mx_quant_kernel(const __grid_constant__ QuantArgs qa) {
  quant_body<kRow, kCol, kGrouped, kMulti, false>(qa, CurParams{nullptr, 0.0f, nullptr});
}

// Current scaling (a separate kernel, so that the MX kernels' parameter block
// stays as it is).
template <bool kRow, bool kCol, bool kGrouped>
__global__ void __launch_bounds__(kThreads, MX_QUANT_MIN_BLOCKS)
    mx_quant_current_kernel(const __grid_constant__ QuantArgs qa, const CurParams cur) {
  quant_body<kRow, kCol, kGrouped, false, true>(qa, cur);
}

// ===========================================================================
// Current scaling: amax of each matrix of a BF16 stack
// ===========================================================================
//
// "DeepSeek-V3 16B FSDP2 MXFP8/HiF8 训练设计" §3 / §8.2: the FP32 scale of a
// tensor comes from the amax of the current tensor (of each leading group for
// a stacked one). One warp per input row at a time, 16-byte loads (four in
// flight per lane), an unsigned max over the BF16 magnitude bits (NaN > Inf >
// finite, as for the blocks), a warp reduction, and one atomic max per warp
// and matrix on the FP32 bit pattern (non-negative floats order like their
// bits). The caller zeroes amax first.
__global__ void __launch_bounds__(256) cur_amax_kernel(const uint16_t* __restrict__ x, int64_t batch, int64_t rows,
                                                       int64_t cols, int64_t ldx, int64_t bstride,
                                                       uint32_t* __restrict__ amax_bits) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t vpr = cols >> 3;  // 16-byte vectors per row (cols % 32 == 0)
  uint32_t m = 0;
  int64_t cur_b = -1;
  auto flush = [&]() {
    const uint32_t r = __reduce_max_sync(0xFFFFFFFFu, half_max(m));
    if (lane == 0 && cur_b >= 0 && r > 0) atomicMax(amax_bits + cur_b, r << 16);
    m = 0;
  };
  for (int64_t gr = warp_id; gr < batch * rows; gr += warps) {
    const int64_t b = gr / rows;
    if (b != cur_b) {  // warp-uniform
      flush();
      cur_b = b;
    }
    const uint4* row = reinterpret_cast<const uint4*>(x + b * bstride + (gr - b * rows) * ldx);
    for (int64_t v = lane; v < vpr; v += 128) {
      uint4 q[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) q[u] = (v + 32 * u < vpr) ? __ldcs(row + v + 32 * u) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        m = __vmaxu2(__vmaxu2(m, __vmaxu2(q[u].x & 0x7FFF7FFFu, q[u].y & 0x7FFF7FFFu)),
                     __vmaxu2(q[u].z & 0x7FFF7FFFu, q[u].w & 0x7FFF7FFFu));
    }
  }
  flush();
}

// ===========================================================================
// FP32 input (weight refresh from the FP32 master)
// ===========================================================================
//
// "DeepSeek-V3 16B FSDP2 MXFP8/HiF8 训练设计" §8.1 and §10: after each
// optimizer step the row and column copies of the weights are produced from the
// FP32 master, so the blocks are formed from the FP32 values themselves (no BF16
// rounding on the way). Same rule and layouts as the BF16 kernel; the tile is
// 128 rows x 64 columns (32 KB), landing as two 32-column boxes in the 128-byte
// swizzled layout (16-byte chunk c of row r at c ^ (r % 8)).

constexpr int kF32Cols = 64;
constexpr int kF32BoxCols = 32;
constexpr int kF32TileBytes = kTileRows * kF32Cols * 4;
constexpr int kF32StageBytes = kF32Cols * kTileRows;  // one E4M3 column-copy tile

// E8M0 code from the largest FP32 magnitude pattern of a block.
__device__ __forceinline__ uint32_t scale_code_f32(uint32_t amax_bits) {
  const int e = static_cast<int>(amax_bits >> 23);  // biased exponent
  if (e == 0xFF) return 0xFFu;                       // block holds Inf or NaN
  return static_cast<uint32_t>(max(e - 127 - 8, -127) + 127);
}

// NaN codes keeping the signs of two FP32 values (a in the low byte).
__device__ __forceinline__ uint32_t nan_pair_f32(uint32_t a, uint32_t b) {
  return (0x7Fu | ((a >> 24) & 0x80u)) | ((0x7Fu | ((b >> 24) & 0x80u)) << 8);
}

// Four FP32 values -> four E4M3 bytes (first value in the low byte).
__device__ __forceinline__ uint32_t quant4_f32(float a, float b, float c, float d, float inv) {
  return cvt_pair(a * inv, b * inv) | (cvt_pair(c * inv, d * inv) << 16);
}

template <bool kRow, bool kCol>
__global__ void __launch_bounds__(kThreads, MX_QUANT_MIN_BLOCKS)
    mx_quant_f32_kernel(const __grid_constant__ CUtensorMap tmap_x, QParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tiles = smem;                                        // kStages x 2 boxes x [128 rows][128 bytes]
  uint8_t* col_stage = tiles + kStages * kF32TileBytes;         // 2 x [64 out rows][128 bytes], swizzled
  uint8_t* col_sc = col_stage + 2 * kF32StageBytes;             // 2 x [64][4] column-copy scales
  uint64_t* full = reinterpret_cast<uint64_t*>(col_sc + 512);
  uint64_t* empty = full + kStages;
  __shared__ volatile int32_t s_abort;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int64_t col_tiles = (p.cols + kF32Cols - 1) / kF32Cols;
  const int64_t row_tiles = (p.rows + kTileRows - 1) / kTileRows;
  const int64_t ntiles = row_tiles * col_tiles * p.batch;
  // Barriers and the tensor-map prefetch touch no global memory: they run
  // before the wait for the previous kernel (as in the BF16 quantiser).
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == kConsumers / 32 && lane == 0) tma_prefetch_desc(&tmap_x);
  // Programmatic dependent launch: let the next kernel on the stream be
  // scheduled, and touch global memory only once the previous one completed.
  pdl_launch_dependents();
  pdl_wait();
  __syncthreads();

  if (warp == kConsumers / 32) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int j = 0;
      int last_phase_issued[kStages];
#pragma unroll
      for (int s = 0; s < kStages; ++s) last_phase_issued[s] = -1;
      for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++j) {
        const int s = j % kStages;
        const uint32_t ph = static_cast<uint32_t>((j / kStages) & 1);
        if (!wait_or_abort(&empty[s], ph ^ 1u, p, &s_abort)) break;
        const int64_t b = t / (row_tiles * col_tiles);
        const int64_t rem = t - b * row_tiles * col_tiles;
        const int64_t rt = rem / col_tiles, ct = rem - rt * col_tiles;
        mbar_arrive_expect_tx(&full[s], kF32TileBytes);
#pragma unroll
        for (int h = 0; h < 2; ++h)
          tma_load_3d(tiles + s * kF32TileBytes + h * (kF32TileBytes / 2), &tmap_x, &full[s],
                      static_cast<int32_t>(ct * kF32Cols + h * kF32BoxCols), static_cast<int32_t>(rt * kTileRows),
                      static_cast<int32_t>(b));
#pragma unroll
        for (int q = 0; q < kStages; ++q)
          if (q == s) last_phase_issued[q] = static_cast<int>(ph);
      }
      if (s_abort) {
#pragma unroll
        for (int q = 0; q < kStages; ++q)
          if (last_phase_issued[q] >= 0) mbar_wait(&full[q], static_cast<uint32_t>(last_phase_issued[q]), p.timeout_ns);
      }
    }
  } else {
    // ----------------------------------------------------------- consumers
    int j = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++j) {
      const int s = j % kStages;
      const uint32_t ph = static_cast<uint32_t>((j / kStages) & 1);
      const int64_t b = t / (row_tiles * col_tiles);
      const int64_t rem = t - b * row_tiles * col_tiles;
      const int64_t rt = rem / col_tiles, ct = rem - rt * col_tiles;
      const int64_t row0 = rt * kTileRows, c0 = ct * kF32Cols;
      const int valid_rows = static_cast<int>(min64(kTileRows, p.rows - row0));
      const int valid_cols = static_cast<int>(min64(kF32Cols, p.cols - c0));
      uint8_t* const row_data = p.row_data + b * p.row_data_bs;
      uint8_t* const row_scale = p.row_scale + b * p.row_scale_bs;
      uint8_t* const col_data = p.col_data + b * p.col_data_bs;
      uint8_t* const col_scale = p.col_scale + b * p.col_scale_bs;
      const uint8_t* tile = tiles + s * kF32TileBytes;
      uint8_t* csc = col_sc + (j & 1) * 256;
      uint8_t* stg = col_stage + (j & 1) * kF32StageBytes;
      const bool ok = !s_abort && wait_or_abort(&full[s], ph, p, &s_abort);

      if (kRow && ok) {
        // ---- row copy: thread = (row r, 32-column block = box blk); the eight
        // lanes of a load phase hold eight consecutive rows -> distinct chunks.
        const int r = (warp & 3) * 32 + lane;
        const int blk = warp >> 2;
        const uint4* src = reinterpret_cast<const uint4*>(tile + blk * (kF32TileBytes / 2)) + r * 8;
        uint4 v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = src[q ^ (r & 7)];
        uint32_t m = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          m = max(max(max(m, v[q].x & 0x7FFFFFFFu), v[q].y & 0x7FFFFFFFu),
                  max(v[q].z & 0x7FFFFFFFu, v[q].w & 0x7FFFFFFFu));
        const uint32_t code = scale_code_f32(m);
        const bool nan_block = (code == 0xFFu);
        const float inv = inv_scale(nan_block ? 0u : code);
        uint32_t o[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          o[q] = quant4_f32(__uint_as_float(v[q].x), __uint_as_float(v[q].y), __uint_as_float(v[q].z),
                            __uint_as_float(v[q].w), inv);
        if (__any_sync(0xFFFFFFFFu, nan_block) && nan_block) {
#pragma unroll
          for (int q = 0; q < 8; ++q) o[q] = nan_pair_f32(v[q].x, v[q].y) | (nan_pair_f32(v[q].z, v[q].w) << 16);
        }
        const int64_t grow = row0 + r;
        if (r < valid_rows && blk * 32 < valid_cols) {
          uint4* dst = reinterpret_cast<uint4*>(row_data + grow * p.cols + c0 + blk * 32);
          dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
          dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
        // Rows past the end were zero-filled by the TMA: they write the zero
        // codes of the scale padding.
        row_scale[scale_offset(grow, (c0 >> 5) + blk, p.row_ka)] = static_cast<uint8_t>(code);
        // A last tile that starts a 4-block scale group alone also writes the
        // zero codes of the group's two remaining (padding) blocks.
        if ((c0 & 127) == 0 && c0 + kF32Cols >= p.cols)
          row_scale[scale_offset(grow, (c0 >> 5) + 2 + blk, p.row_ka)] = 0;
      }

      if constexpr (kCol) {
        if (ok) {
          // ---- column copy: thread = (column c, 32-row block rb)
          const int c = tid & 63;
          const int rb = tid >> 6;
          const uint32_t* src = reinterpret_cast<const uint32_t*>(tile + (c >> 5) * (kF32TileBytes / 2)) +
                                rb * 32 * 32 + (c & 3);
          const int cc = (c & 31) >> 2;
          uint32_t w[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) w[i] = src[i * 32 + ((cc ^ (i & 7)) << 2)];
          mbar_arrive(&empty[s]);  // this thread is done with the tile
          uint32_t m = 0;
#pragma unroll
          for (int i = 0; i < 32; ++i) m = max(m, w[i] & 0x7FFFFFFFu);
          const uint32_t code = scale_code_f32(m);
          const bool nan_block = (code == 0xFFu);
          const float inv = inv_scale(nan_block ? 0u : code);
          uint32_t o[8];
#pragma unroll
          for (int q = 0; q < 8; ++q)
            o[q] = quant4_f32(__uint_as_float(w[4 * q]), __uint_as_float(w[4 * q + 1]),
                              __uint_as_float(w[4 * q + 2]), __uint_as_float(w[4 * q + 3]), inv);
          if (__any_sync(0xFFFFFFFFu, nan_block) && nan_block) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              o[q] = nan_pair_f32(w[4 * q], w[4 * q + 1]) | (nan_pair_f32(w[4 * q + 2], w[4 * q + 3]) << 16);
          }
          csc[c * 4 + rb] = static_cast<uint8_t>(code);
          // Output row c, 16-byte chunks 2rb and 2rb+1, chunk q at q ^ (c % 8).
          *reinterpret_cast<uint4*>(stg + c * 128 + (((2 * rb) ^ (c & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(stg + c * 128 + (((2 * rb + 1) ^ (c & 7)) << 4)) =
              make_uint4(o[4], o[5], o[6], o[7]);
        }
        consumers_sync();
        if (ok) {
#pragma unroll
          for (int it = 0; it < (kF32Cols * 8) / kConsumers; ++it) {
            const int idx = it * kConsumers + tid;
            const int o = idx >> 3;
            const int q = idx & 7;
            if (o < valid_cols && q * 16 < valid_rows)
              *reinterpret_cast<uint4*>(col_data + (c0 + o) * p.col_pitch + row0 + q * 16) =
                  *reinterpret_cast<const uint4*>(stg + o * 128 + ((q ^ (o & 7)) << 4));
          }
          if (tid < kF32Cols)
            *reinterpret_cast<uint32_t*>(col_scale + scale_offset(c0 + tid, row0 >> 5, p.col_ka)) =
                *reinterpret_cast<const uint32_t*>(csc + tid * 4);
          // Likewise the padding rows of a 128-row scale group that the last
          // column tile starts alone.
          else if (tid < 2 * kF32Cols && (c0 & 127) == 0 && c0 + kF32Cols >= p.cols)
            *reinterpret_cast<uint32_t*>(col_scale + scale_offset(c0 + tid, row0 >> 5, p.col_ka)) = 0u;
        }
      } else {
        if (ok) mbar_arrive(&empty[s]);
      }
    }
  }
}

// ===========================================================================
// Variant recipe: DeepSeek-V3 blockwise FP8 (FP32 multipliers per block)
// ===========================================================================
//
// "浮点格式、数值稳定性与混合精度" §七.2-§七.3: a block's multiplier is
// s = 448 / amax and its elements are E4M3(s * x); activations use 1 x 128
// blocks along the row, weights 128 x 128 blocks. Both steps are FP32 IEEE
// operations (division and product correctly rounded) followed by the
// round-to-nearest-even satfinite E4M3 conversion; an all-zero block takes
// s = 1.

__device__ __forceinline__ float blockwise_s(float amax) { return amax > 0.0f ? 448.0f / amax : 1.0f; }

// Four BF16 values (two words) times s -> four E4M3 bytes.
__device__ __forceinline__ uint32_t blockwise_quad(uint32_t w0, uint32_t w1, float s) {
  return cvt_pair(__fmul_rn(lo_f(w0), s), __fmul_rn(hi_f(w0), s)) |
         (cvt_pair(__fmul_rn(lo_f(w1), s), __fmul_rn(hi_f(w1), s)) << 16);
}

// 1 x 128 blocks: a half-warp per block (lane = 8 consecutive elements, one
// 16-byte load), each warp on two consecutive blocks of a row per step.
// s is stored transposed, scale[kb * rows + r].
__global__ void __launch_bounds__(256) fp8_quant_1x128_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows,
                                                              int64_t cols, int64_t ldx, uint8_t* __restrict__ data,
                                                              float* __restrict__ scale) {
  // Programmatic dependent launch: touch global memory only once the previous
  // kernel on the stream has completed; let the next one be scheduled once
  // this CTA's work is done (its small CTAs waiting beside a running grid
  // would take issue slots from it).
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int hl = lane & 15;
  const int64_t kbs = cols / 128;
  const int64_t nblocks = rows * kbs;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t b2 = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); 2 * b2 < nblocks;
       b2 += warps) {
    const int64_t b = 2 * b2 + (lane >> 4);  // this half-warp's block (kbs is even or the row ends)
    const bool in = b < nblocks;
    const int64_t r = in ? b / kbs : 0, kb = in ? b - (b / kbs) * kbs : 0;
    const uint4 v = in ? *reinterpret_cast<const uint4*>(x + r * ldx + kb * 128 + hl * 8) : make_uint4(0u, 0u, 0u, 0u);
    uint32_t m = max(max(half_max(v.x & 0x7FFF7FFFu), half_max(v.y & 0x7FFF7FFFu)),
                     max(half_max(v.z & 0x7FFF7FFFu), half_max(v.w & 0x7FFF7FFFu)));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));  // within the half-warp
    const float s = blockwise_s(__uint_as_float(m << 16));
    if (in) {
      *reinterpret_cast<uint2*>(data + r * cols + kb * 128 + hl * 8) =
          make_uint2(blockwise_quad(v.x, v.y, s), blockwise_quad(v.z, v.w, s));
      if (hl == 0) scale[kb * rows + r] = s;
    }
  }
  pdl_launch_dependents();
}

// 128 x 128 blocks: one CTA per block; thread t holds 64 elements of row t/2.
__global__ void __launch_bounds__(256) fp8_quant_128x128_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows,
                                                                int64_t cols, int64_t ldx,
                                                                uint8_t* __restrict__ data,
                                                                float* __restrict__ scale) {
  pdl_wait();  // as in fp8_quant_1x128_kernel
  __shared__ uint32_t warp_max[8];
  const int tid = threadIdx.x;
  const int64_t kbs = cols / 128;
  const int64_t rbs = (rows + 127) / 128;
  for (int64_t b = blockIdx.x; b < rbs * kbs; b += gridDim.x) {
    const int64_t rb = b / kbs, kb = b - rb * kbs;
    const int64_t r = rb * 128 + (tid >> 1);
    const bool in = r < rows;
    uint4 v[8];  // 64 BF16 values of row r: columns (tid & 1) * 64 .. + 63 of the block
    uint32_t m = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      v[q] = in ? *reinterpret_cast<const uint4*>(x + r * ldx + kb * 128 + (tid & 1) * 64 + q * 8)
                : make_uint4(0u, 0u, 0u, 0u);
      m = max(m, max(max(half_max(v[q].x & 0x7FFF7FFFu), half_max(v[q].y & 0x7FFF7FFFu)),
                     max(half_max(v[q].z & 0x7FFF7FFFu), half_max(v[q].w & 0x7FFF7FFFu))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((tid & 31) == 0) warp_max[tid >> 5] = m;
    __syncthreads();
    uint32_t bm = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) bm = max(bm, warp_max[w]);
    __syncthreads();  // warp_max is rewritten by the next block
    const float s = blockwise_s(__uint_as_float(bm << 16));
    if (in) {
      uint4* dst = reinterpret_cast<uint4*>(data + r * cols + kb * 128 + (tid & 1) * 64);
#pragma unroll
      for (int q = 0; q < 8; q += 2)
        dst[q >> 1] = make_uint4(blockwise_quad(v[q].x, v[q].y, s), blockwise_quad(v[q].z, v[q].w, s),
                                 blockwise_quad(v[q + 1].x, v[q + 1].y, s), blockwise_quad(v[q + 1].z, v[q + 1].w, s));
    }
    if (tid == 0) scale[rb * kbs + kb] = s;
  }
  pdl_launch_dependents();
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

template <bool R, bool C, bool G, bool M = false, bool kCur = false>
mx_status launch_one(const QuantArgs& qa, int64_t tiles_upper, cudaStream_t s, CurParams cur = CurParams{}) {
  const size_t smem = 1024 + static_cast<size_t>(kStages) * kTileBytes + 2 * kColStageBytes + 1024 + 2 * kStages * 8 +
                      (G ? 2 * (kMaxGroups + 1) * sizeof(int32_t) : 0);
  if constexpr (kCur) {
    auto kern = mx_quant_current_kernel<R, C, G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_status(e, "cudaFuncSetAttribute(quant smem)");
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
    if (e != cudaSuccess) return cuda_status(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    const int64_t grid =
        std::max<int64_t>(1, std::min<int64_t>(tiles_upper, static_cast<int64_t>(std::max(per_sm, 1)) * sm_count()));
    return cuda_status(launch_kernel(kern, static_cast<unsigned>(grid), kThreads, smem, s, 1, qa, cur),
                       "mx_quantize_current launch");
  }
  auto kern = mx_quant_kernel<R, C, G, M>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_status(e, "cudaFuncSetAttribute(quant smem)");
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
  if (e != cudaSuccess) return cuda_status(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
  const int64_t grid =
      std::max<int64_t>(1, std::min<int64_t>(tiles_upper, static_cast<int64_t>(std::max(per_sm, 1)) * sm_count()));
  return cuda_status(launch_kernel(kern, static_cast<unsigned>(grid), kThreads, smem, s, 1, qa), "mx_quantize launch");
}

template <bool R, bool C>
mx_status launch_f32_one(const CUtensorMap& map, const QParams& p, int64_t tiles, cudaStream_t s) {
  const size_t smem = 1024 + static_cast<size_t>(kStages) * kF32TileBytes + 2 * kF32StageBytes + 512 + 2 * kStages * 8;
  auto kern = mx_quant_f32_kernel<R, C>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_status(e, "cudaFuncSetAttribute(quant f32 smem)");
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
  if (e != cudaSuccess) return cuda_status(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
  const int64_t grid =
      std::max<int64_t>(1, std::min<int64_t>(tiles, static_cast<int64_t>(std::max(per_sm, 1)) * sm_count()));
  return cuda_status(launch_kernel(kern, static_cast<unsigned>(grid), kThreads, smem, s, 1, map, p),
                     "mx_quantize_f32 launch");
}

// FP32 input: [batch, rows, cols] through 32-column boxes in the 128-byte swizzle.
mx_status launch_f32(const QuantLaunch& q, const QParams& p, bool do_row, bool do_col, cudaStream_t s) {
  const int64_t tiles = (q.rows + kTileRows - 1) / kTileRows * ((q.cols + kF32Cols - 1) / kF32Cols) * q.batch;
  if (tiles == 0) return MX_OK;
  EncodeTiledFn enc = encode_fn();
  if (!enc) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return MX_ERR_CUDA;
  }
  CUtensorMap map;
  std::memset(&map, 0, sizeof(map));
  const int64_t bstride = q.batch > 1 ? q.x_batch_stride : q.rows * q.ldx;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(q.cols), static_cast<cuuint64_t>(q.rows),
                        static_cast<cuuint64_t>(q.batch)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(q.ldx * 4), static_cast<cuuint64_t>(bstride * 4)};
  cuuint32_t box[3] = {kF32BoxCols, kTileRows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(q.x), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled (FP32 quantiser input) failed (%d)", static_cast<int>(r));
    return MX_ERR_CUDA;
  }
  if (do_row && do_col) return launch_f32_one<true, true>(map, p, tiles, s);
  if (do_row) return launch_f32_one<true, false>(map, p, tiles, s);
  return launch_f32_one<false, true>(map, p, tiles, s);
}

}  // namespace

mx_status launch_quantize_blockwise(const void* x, int64_t rows, int64_t cols, int64_t ldx, int block, void* data,
                                    float* scale, cudaStream_t s) {
  const int64_t blocks = block == 1 ? rows * (cols / 128) : (rows + 127) / 128 * (cols / 128);
  if (blocks == 0) return MX_OK;
  if (block == 1) {
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((blocks + 15) / 16, 16LL * sm_count()));
    return cuda_status(launch_kernel(fp8_quant_1x128_kernel, static_cast<unsigned>(grid), 256, 0, s, 1,
                                     static_cast<const __nv_bfloat16*>(x), rows, cols, ldx,
                                     static_cast<uint8_t*>(data), scale),
                       "mx_quantize_fp8_blockwise launch");
  } else {
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(blocks, 8LL * sm_count()));
    return cuda_status(launch_kernel(fp8_quant_128x128_kernel, static_cast<unsigned>(grid), 256, 0, s, 1,
                                     static_cast<const __nv_bfloat16*>(x), rows, cols, ldx,
                                     static_cast<uint8_t*>(data), scale),
                       "mx_quantize_fp8_blockwise launch");
  }
}

namespace {

QParams make_qparams(const QuantLaunch& q) {
  QParams p;
  p.rows = q.rows;
  p.cols = q.cols;
  p.row_data = static_cast<uint8_t*>(q.row_data);
  p.row_scale = static_cast<uint8_t*>(q.row_scale);
  p.col_data = static_cast<uint8_t*>(q.col_data);
  p.col_scale = static_cast<uint8_t*>(q.col_scale);
  p.offsets = q.offsets;
  p.n_groups = q.n_groups;
  p.col_pitch = q.col_pitch;
  p.row_ka = (q.cols + 127) / 128;
  p.col_ka = (q.col_pitch + 127) / 128;
  p.dev_status = q.dev_status;
  p.batch = q.batch;
  p.row_data_bs = q.rows * q.cols;
  p.row_scale_bs = static_cast<int64_t>(mx_scale_bytes(q.rows, q.cols));
  p.col_data_bs = q.cols * q.col_pitch;
  p.col_scale_bs = static_cast<int64_t>(mx_scale_bytes(q.cols, q.col_pitch));
  p.timeout_ns = wait_timeout_ns();
  return p;
}

// [batch, rows, cols] view of a BF16 input (a single matrix is a batch of one),
// 64-column boxes in the 128-byte swizzle.
mx_status make_bf16_input_map(const QuantLaunch& q, CUtensorMap* map) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return MX_ERR_CUDA;
  }
  std::memset(map, 0, sizeof(*map));
  const int64_t bstride = q.batch > 1 ? q.x_batch_stride : q.rows * q.ldx;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(q.cols), static_cast<cuuint64_t>(q.rows),
                        static_cast<cuuint64_t>(q.batch)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(q.ldx * 2), static_cast<cuuint64_t>(bstride * 2)};
  cuuint32_t box[3] = {kHalfCols, kTileRows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q.x), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled (quantiser input) failed (%d)", static_cast<int>(r));
    return MX_ERR_CUDA;
  }
  return MX_OK;
}

mx_status launch_by_axis(const QuantArgs& qa, int64_t tiles, bool do_row, bool do_col, bool grouped, cudaStream_t s) {
  if (grouped)
    return do_row ? launch_one<true, true, true>(qa, tiles, s) : launch_one<false, true, true>(qa, tiles, s);
  if (qa.n > 1) {
    if (do_row && do_col) return launch_one<true, true, false, true>(qa, tiles, s);
    if (do_row) return launch_one<true, false, false, true>(qa, tiles, s);
    return launch_one<false, true, false, true>(qa, tiles, s);
  }
  if (do_row && do_col) return launch_one<true, true, false>(qa, tiles, s);
  if (do_row) return launch_one<true, false, false>(qa, tiles, s);
  return launch_one<false, true, false>(qa, tiles, s);
}

}  // namespace

mx_status launch_current_amax(const QuantLaunch& q, float* amax, cudaStream_t s) {
  mx_status st = cuda_status(cudaMemsetAsync(amax, 0, static_cast<size_t>(q.batch) * sizeof(float), s),
                             "cudaMemsetAsync(amax)");
  if (st != MX_OK || q.rows == 0 || q.cols == 0) return st;
  const int64_t bstride = q.batch > 1 ? q.x_batch_stride : q.rows * q.ldx;
  const int64_t warps_needed = q.batch * q.rows;
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((warps_needed + 7) / 8, 8LL * sm_count()));
  return cuda_status(launch_kernel(cur_amax_kernel, static_cast<unsigned>(grid), 256, 0, s, 1,
                                   static_cast<const uint16_t*>(q.x), q.batch, q.rows, q.cols, q.ldx, bstride,
                                   reinterpret_cast<uint32_t*>(amax)),
                     "current amax launch");
}

mx_status launch_quantize_current(const QuantLaunch& q, const float* amax, float format_max, float* scale,
                                  bool do_row, bool do_col, cudaStream_t s) {
  const QParams p = make_qparams(q);
  const bool grouped = q.offsets != nullptr && do_col;
  const int64_t col_tiles = (q.cols + kTileCols - 1) / kTileCols;
  int64_t row_tiles = (q.rows + kTileRows - 1) / kTileRows;
  if (grouped) row_tiles += q.n_groups;  // upper bound of sum ceil(m_e / 128)
  QuantArgs qa;
  std::memset(&qa, 0, sizeof(qa));
  mx_status st = make_bf16_input_map(q, &qa.map[0]);
  if (st != MX_OK) return st;
  qa.p[0] = p;
  qa.n = 1;
  const CurParams cur{amax, format_max, scale};
  // an empty matrix still gets its scale (1): one tile's worth of launch
  const int64_t tiles = std::max<int64_t>(1, row_tiles * col_tiles * q.batch);
  qa.tile0[0] = 0;
  qa.tile0[1] = row_tiles * col_tiles * q.batch;
  if (grouped)
    return do_row ? launch_one<true, true, true, false, true>(qa, tiles, s, cur)
                  : launch_one<false, true, true, false, true>(qa, tiles, s, cur);
  if (do_row && do_col) return launch_one<true, true, false, false, true>(qa, tiles, s, cur);
  if (do_row) return launch_one<true, false, false, false, true>(qa, tiles, s, cur);
  return launch_one<false, true, false, false, true>(qa, tiles, s, cur);
}

mx_status launch_quantize(const QuantLaunch& q, bool do_row, bool do_col, cudaStream_t s) {
  const QParams p = make_qparams(q);
  const bool grouped = q.offsets != nullptr && do_col;
  if (grouped && q.n_groups > kMaxGroups) {
    set_error("mx_quantize: at most %d groups", kMaxGroups);
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  if (q.x_f32) return launch_f32(q, p, do_row, do_col, s);
  const int64_t col_tiles = (q.cols + kTileCols - 1) / kTileCols;
  int64_t row_tiles = (q.rows + kTileRows - 1) / kTileRows;
  if (grouped) row_tiles += q.n_groups;  // upper bound of sum ceil(m_e / 128)
  if (row_tiles == 0 || col_tiles == 0) return MX_OK;
  QuantArgs qa;
  std::memset(&qa, 0, sizeof(qa));
  mx_status st = make_bf16_input_map(q, &qa.map[0]);
  if (st != MX_OK) return st;
  qa.p[0] = p;
  qa.n = 1;
  const int64_t tiles = row_tiles * col_tiles * q.batch;
  qa.tile0[0] = 0;
  qa.tile0[1] = tiles;
  return launch_by_axis(qa, tiles, do_row, do_col, grouped, s);
}

mx_status launch_quantize_multi(const QuantLaunch* qs, int n, bool do_row, bool do_col, cudaStream_t s) {
  if (n < 1 || n > kMaxTensors) {
    set_error("mx_quantize_multi: 1 to %d tensors", kMaxTensors);
    return MX_ERR_INVALID_ARG;
  }
  QuantArgs qa;
  std::memset(&qa, 0, sizeof(qa));
  int64_t tiles = 0;
  int m = 0;
  for (int i = 0; i < n; ++i) {
    const QuantLaunch& q = qs[i];
    const int64_t t = (q.rows + kTileRows - 1) / kTileRows * ((q.cols + kTileCols - 1) / kTileCols);
    if (t == 0) continue;  // an empty matrix has nothing to write
    mx_status st = make_bf16_input_map(q, &qa.map[m]);
    if (st != MX_OK) return st;
    qa.p[m] = make_qparams(q);
    qa.tile0[m] = tiles;
    tiles += t;
    ++m;
  }
  if (m == 0) return MX_OK;
  qa.n = m;
  qa.tile0[m] = tiles;
  return launch_by_axis(qa, tiles, do_row, do_col, false, s);
}

}  // namespace mx
