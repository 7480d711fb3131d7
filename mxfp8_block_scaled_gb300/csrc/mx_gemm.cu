// mx_gemm.cu - block-scaled MXFP8 GEMM and grouped GEMM on the sm_103a
// tensor cores (tcgen05.mma kind::mxf8f6f4 with UE8M0 block scales).
//
// Computes C[M, N] = A[M, K] . B[N, K]^T with both operands K-major E4M3
// codes and one E8M0 scale per 32 elements along K, FP32 accumulation in
// tensor memory and a BF16 round-to-nearest-even epilogue. This is the GEMM of
// the direction table in "DeepSeek-V3 16B FSDP2 MXFP8/HiF8 训练设计" §8
// (fprop / dgrad / wgrad all reduce to A . B^T once column copies are stored
// transposed) and of §5.2 / §13.4 for the routed experts (grouped GEMM over
// group_list offsets); FP32 accumulation with BF16 output follows
// "浮点格式、数值稳定性与混合精度" §五.1. The block scales vary along K, so
// they are applied inside the accumulation (by the MMA itself, per 32-K step),
// not in the epilogue (same page, §七.3).
//
// Two kernels share the tile bookkeeping and the epilogue:
//
// mx_gemm_kernel (one CTA per SM, persistent over 128 x BN output tiles):
//   warp 0      TMA producer: A and B tiles (128-byte swizzled boxes of 128 K
//               elements) and the 512-byte scale atoms of each K block into a
//               ring of shared-memory stages, completion on mbarriers.
//   warp 1      allocates tensor memory; lane 0 issues, per K block, four
//               K=32 MMAs (scale byte selector = K step), then commits the
//               stage back to the producer; after the last K block it commits
//               the accumulator.
//   warps 2-9   epilogue: pull the tile out of TMEM with tcgen05.ld, release
//               the accumulator at once, convert to BF16 and write 32 x 32
//               boxes through swizzled shared memory with TMA stores.
//   warp 10     scale copier: per K block, one tcgen05.cp per scale atom into
//               the stage's TMEM slot, committed to a barrier the MMA issuer
//               waits on. Issued from the MMA thread itself these copies sit
//               in its instruction stream between the MMAs and cost ~10% of
//               the tensor-pipe time; from a warp of their own they overlap.
//
// mx_gemm_pair_kernel (CTA pairs = clusters of two, cta_group::2; the kernel
// for every shape that fills the GPU with 256 x 256 tiles):
//   a 256 x 256 tile per pair. Each CTA loads its 128 rows of A and its half
//   of B (so a stage is 32 KB instead of 48 KB and six stages fit), the even
//   CTA issues the pair-wide MMAs (M = 256) and scale copies, and every
//   completion is multicast to both CTAs. The MMA issuer waits once per stage,
//   on the copier's barrier (which follows the stage's full barrier); in cycle
//   traces its own instruction stream, not the operand feed, sets the stage
//   time. Variants: dense (optionally several independent GEMMs per launch,
//   and a split tail for few-tile long-K shapes), rows-ragged grouped (A scale
//   atoms gathered by warp 11 for tiles that start at any row; the SwiGLU
//   epilogue writing BF16 or the MX copies of its output), K-ragged grouped,
//   and tensor-scaled (plain E4M3 MMAs, two accumulators, no scale copies).
//
// Every mbarrier wait is bounded in wall time; on expiry the CTA records
// MX_ERR_TIMEOUT in dev_status, drains its own copies and MMAs, frees its
// tensor memory and returns.
//
// Grouped variants of the single-CTA kernel (small grids): rows-ragged
// (fprop/dgrad over contiguous token ranges per expert; A tiles start at
// arbitrary rows, so the producer warp gathers their scale atoms with
// cp.async) and contraction-ragged (wgrad; per-expert K segments padded to
// 128, one output matrix per expert, experts with most K scheduled first; an
// empty expert writes zeros).

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <mutex>
#include <queue>
#include <utility>
#include <vector>

#include "mx_codec.cuh"
#include "mx_internal.h"
#include "mx_ptx.cuh"

namespace mx {
namespace {

constexpr int kBM = 128;       // tile rows per CTA (MMA M of one CTA)
constexpr int kBK = 128;       // K elements (= bytes) per stage: four K=32 MMAs
constexpr int kThreads = 352;  // producer, MMA, 8 epilogue warps, scale copier
constexpr int kCopierWarp = 10;
constexpr int kPairThreads = 384;  // the pair kernel adds a scale-gather warp
constexpr int kGatherWarp = 11;
constexpr int kEpiThreads = 256;
constexpr int kMaxGroups = MX_MAX_GROUPS;
constexpr uint32_t kTmemCols = 512;
constexpr int kEpiWarpBytes = 32 * 64;  // one 32-row x 32-column BF16 box per epilogue warp
constexpr int kEpiBytes = 8 * kEpiWarpBytes;

// Epilogue write-out: 0 = TMA tensor stores from the staging box (asynchronous:
// the warp stages the next box while the previous one drains; 2-8% faster on
// GB300, most for short contractions where the output write dominates),
// 1 = shared-memory staging + coalesced 16-byte stores by the warp itself.
#ifndef MX_EPI_MODE
#define MX_EPI_MODE 0
#endif

template <int BN>
struct Cfg {
  // BN = 256 leaves no tensor memory for a second accumulator next to the
  // per-stage scale columns; BN = 128 double-buffers the accumulator so the
  // epilogue of one tile overlaps the MMAs of the next.
  static constexpr int kStages = (BN == 128) ? 6 : 4;
  static constexpr int kAcc = (BN == 256) ? 1 : 2;
  static constexpr int kABytes = kBM * kBK;
  static constexpr int kBBytes = BN * kBK;
  static constexpr int kSfbAtoms = (BN + 127) / 128;
  static constexpr int kSfbBytes = kSfbAtoms * 512;
  static constexpr int kSfCols = 4 + 4 * kSfbAtoms;     // TMEM columns of one stage's scales
  static constexpr uint32_t kSfCol0 = kAcc * BN;        // first scale column
  static_assert(kSfCol0 + kStages * kSfCols <= kTmemCols, "TMEM budget");
  // B tiles must start on a 128-row scale atom, so the atoms load as they are.
  static_assert(BN % 128 == 0, "tile width must be a multiple of 128");
  static constexpr int kBarBytes = (3 * kStages + 2 * kAcc + 2) * 8 + 16;
  static constexpr int kGroupBytes = 3 * (kMaxGroups + 1) * 4;
  __host__ __device__ static constexpr size_t smem_bytes(bool grouped) {
    return 1024 + static_cast<size_t>(kStages) * (kABytes + kBBytes + 512 + kSfbBytes) + kEpiBytes + kBarBytes +
           (grouped ? kGroupBytes : 0);
  }
};

// CTA-pair configurations: 256 x 256 tiles. Each CTA loads its 128 rows of A
// and 128 rows of B per stage (plus, with block scales, its A scale atom and
// both B scale atoms), and its tensor memory holds its 128 rows of the
// accumulator.
//   Block scales: one 256-column accumulator; the six stages' scale slots
//     take 72 of the remaining columns, so the next tile's MMAs wait for the
//     epilogue to drain the accumulator.
//   kTS (one FP32 scale per tensor or per group, no block scales): two
//     256-column accumulators take all 512 columns, so the epilogue drains
//     one while the MMAs fill the other; no scale slots, no scale copies.
#ifndef MX_PAIR_STAGES
#define MX_PAIR_STAGES 6
#endif
#ifndef MX_PAIR_EPI_BUFS
#define MX_PAIR_EPI_BUFS 1
#endif
template <int BN_, bool kTS_, bool kGrouped_>
struct PairCfgT {
  static constexpr int BN = BN_;
  static constexpr bool kTS = kTS_;
  static_assert(BN == 256, "pair tiles are 256 wide");
  static constexpr int kStages = MX_PAIR_STAGES;
  static constexpr int kEpiBufs = MX_PAIR_EPI_BUFS;  // staging boxes per epilogue warp
  static constexpr int kABytes = kBM * kBK;
  static constexpr int kBBytes = (BN / 2) * kBK;
  static constexpr int kSfaBytes = kTS ? 0 : 512;
  static constexpr int kSfbBytes = kTS ? 0 : 2 * 512;
  static constexpr int kStageTx = kABytes + kBBytes + kSfaBytes + kSfbBytes;  // bytes of one CTA's stage
  static constexpr int kSfCols = kTS ? 0 : 4 + 8;
  static constexpr int kAcc = (2 * BN + kStages * kSfCols <= static_cast<int>(kTmemCols)) ? 2 : 1;
  static constexpr uint32_t kSfCol0 = kAcc * BN;
  static_assert(kSfCol0 + kStages * kSfCols <= kTmemCols, "TMEM budget");
  static constexpr int kBarBytes = (4 * kStages + 6) * 8 + 16 + 2 * MX_MAX_GEMM_MULTI * 4;  // + schedule words
  static constexpr int kGroupBytes = 3 * (kMaxGroups + 1) * 4;
  __host__ __device__ static constexpr size_t smem_bytes() {
    return 1024 + static_cast<size_t>(kStages) * kStageTx + kEpiBufs * kEpiBytes + kBarBytes +
           (kGrouped_ ? kGroupBytes : 0);
  }
};
// The configuration bookkeeping that does not depend on the tile width.
using PairCfg = PairCfgT<256, false, false>;
static_assert(PairCfgT<256, false, true>::smem_bytes() <= 232448, "shared memory");
static_assert(PairCfgT<256, true, true>::smem_bytes() <= 232448, "shared memory");

struct GParams {
  const uint8_t* a_scale;
  const uint8_t* b_scale;
  int64_t M, N, K;
  int64_t n_out;          // columns of C (N, or N/2 behind the SwiGLU epilogue)
  int64_t ka;             // scale-column atoms along K: ceil(K/128)
  int64_t a_ra;           // row atoms of A's scales
  int64_t b_ra;           // row atoms of B's scales (per expert when grouped by rows)
  int64_t b_rows_group;   // rows of one expert's B (grouped by rows)
  int64_t b_scale_stride; // bytes of one expert's B scales (grouped by rows)
  __nv_bfloat16* c;
  int64_t ldc;
  int64_t c_group_stride; // elements between experts' outputs (grouped by K)
  int32_t c_vec;          // 1: every output row start is 16-byte aligned (16-byte stores)
  int32_t c_tma;          // 1: output tiles leave through TMA stores (needs c_vec)
  int32_t n_fast;         // 1: consecutive tiles walk N first (the CTAs sharing an A tile run together)
  const int64_t* offsets;
  int n_groups;
  int* dev_status;
  uint64_t timeout_ns;
  // Dense pair kernel, split tail (sk_w > 0): tiles [sk_first, mu*nt) are the
  // last partial wave. Their K blocks, laid end to end (sk_total of them), are
  // cut into sk_slots runs of sk_w blocks, one run per pair of SMs; a run
  // covers at most two tiles (two segments), and each segment leaves an FP32
  // partial tile in ws for the reduction kernel.
  int64_t sk_first;
  int64_t sk_total;
  int32_t sk_w;
  int32_t sk_slots;
  float* ws;
  // One FP32 scale per tensor (kTS kernels): C = (A . B^T) * ts_a[0] * ts_b[g]
  // with g the tile's expert for rows-ragged grouped GEMMs, else 0.
  const float* ts_a;
  const float* ts_b;
  // Rows-ragged SwiGLU with its output quantised in the epilogue: the column
  // capacity of the per-expert column copy (0 otherwise; the output pointers
  // are in the launch's QOut).
  int64_t q_cap;
};

// Outputs of the quantised SwiGLU epilogue, exactly as mx_quantize writes them
// from the BF16 output: the MX row copy [M, n_out] with its scales and the
// per-expert column copy [n_out, q_cap] with its scales.
struct QOut {
  uint8_t* row_data;
  uint8_t* row_scale;
  uint8_t* col_data;
  uint8_t* col_scale;
};

// One segment's partial tile in the workspace: [unit][cta of the pair][epilogue
// warp][32 float4 columns][32 lanes], so each warp store covers 512 bytes.
constexpr int64_t kPartialFloats = 2LL * 8 * 32 * 32 * 4;  // 256 x 256

struct Tile {
  int64_t m0, n0;      // output tile origin (this CTA's rows) within the (per-expert) C
  int64_t a_row;       // first row of A to load
  int64_t b_row;       // first row of B's 2-D view to load
  int64_t k_atom0;     // first 128-K block of the contraction
  int32_t nkb;         // number of 128-K blocks
  int32_t valid_m;     // rows of the tile that exist (may be <= 0 for a pair's spare tile)
  int32_t group;       // expert (grouped kinds)
  int32_t part;        // -1: whole tile; >= 0: split-tail segment (workspace unit); -2: empty segment
  int32_t n_mma;       // pair tiles: the MMA's N (the tile width, or less for the last columns of C)
  const uint8_t* sfb;  // base of B's scales for this tile's expert
  __nv_bfloat16* cbase;  // C element (m0, n0)
};

struct GroupInfo {
  int32_t* off;    // [E+1] row offsets
  int32_t* tile;   // [E+1] rows-ragged: m-tile prefix; K-ragged: padded 128-block prefix
  int32_t* order;  // K-ragged: [E] experts by decreasing K; rows-ragged: [E+1] 128-padded row prefix
  int32_t total;   // rows-ragged: sum of m-tiles; K-ragged: sum of padded blocks
};

__device__ __forceinline__ int32_t last_le(const int32_t* v, int n, int32_t x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (v[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <int BN, int KIND>
__device__ __forceinline__ int64_t num_tiles(const GParams& p, const GroupInfo& g) {
  const int64_t nt = (p.N + BN - 1) / BN;
  const int64_t mt = (p.M + kBM - 1) / kBM;
  if (KIND == GEMM_DENSE) return mt * nt;
  if (KIND == GEMM_GROUPED_M) return static_cast<int64_t>(g.total) * nt;
  return static_cast<int64_t>(p.n_groups) * mt * nt;
}

template <int BN, int KIND>
__device__ __forceinline__ Tile get_tile(const GParams& p, const GroupInfo& g, int64_t t) {
  Tile ti;
  ti.part = -1;
  const int64_t nt = (p.N + BN - 1) / BN;
  const int64_t mt = (p.M + kBM - 1) / kBM;
  if (KIND == GEMM_DENSE) {
    const int64_t mb = p.n_fast ? t / nt : t % mt;
    const int64_t nb = p.n_fast ? t % nt : t / mt;
    ti.m0 = mb * kBM;
    ti.n0 = nb * BN;
    ti.a_row = ti.m0;
    ti.b_row = ti.n0;
    ti.k_atom0 = 0;
    ti.nkb = static_cast<int32_t>((p.K + kBK - 1) / kBK);
    ti.valid_m = static_cast<int32_t>(min64(kBM, p.M - ti.m0));
    ti.group = 0;
    ti.sfb = p.b_scale;
    ti.cbase = p.c + ti.m0 * p.ldc + ti.n0;
  } else if (KIND == GEMM_GROUPED_M) {
    const int64_t T = g.total;
    const int32_t u = static_cast<int32_t>(p.n_fast ? t / nt : t % T);
    const int64_t nb = p.n_fast ? t % nt : t / T;
    const int e = last_le(g.tile, p.n_groups, u);
    ti.m0 = static_cast<int64_t>(g.off[e]) + static_cast<int64_t>(u - g.tile[e]) * kBM;
    ti.n0 = nb * BN;
    ti.a_row = ti.m0;
    ti.b_row = static_cast<int64_t>(e) * p.b_rows_group + ti.n0;
    ti.k_atom0 = 0;
    ti.nkb = static_cast<int32_t>((p.K + kBK - 1) / kBK);
    ti.valid_m = static_cast<int32_t>(min64(kBM, g.off[e + 1] - ti.m0));
    ti.group = e;
    ti.sfb = p.b_scale + static_cast<int64_t>(e) * p.b_scale_stride;
    ti.cbase = p.c + ti.m0 * p.ldc + ti.n0;
  } else {
    const int64_t per = mt * nt;
    const int e = g.order[t / per];
    const int64_t rem = t % per;
    const int64_t mb = rem % mt, nb = rem / mt;
    ti.m0 = mb * kBM;
    ti.n0 = nb * BN;
    ti.a_row = ti.m0;
    ti.b_row = ti.n0;
    ti.k_atom0 = g.tile[e];
    ti.nkb = g.tile[e + 1] - g.tile[e];
    ti.valid_m = static_cast<int32_t>(min64(kBM, p.M - ti.m0));
    ti.group = e;
    ti.sfb = p.b_scale;
    ti.cbase = p.c + static_cast<int64_t>(e) * p.c_group_stride + ti.m0 * p.ldc + ti.n0;
  }
  return ti;
}

// Pair tiles: t enumerates (pair of M tiles, N tile); the CTA's rank in its
// cluster picks the M tile, both CTAs share the BN-wide N tile. K-ragged
// grouped: experts in decreasing-K order, each expert's pair tiles M-fastest.
// The MMA width of a pair tile starting at column n0: the tile width, or, for
// the last tile of a C whose width is not a multiple of it, the columns left
// rounded up to 32 (each CTA then holds a multiple of 16 rows of B). The MMAs
// take time in proportion to their N, so a narrow last tile costs only its
// own columns.
template <int BN>
__device__ __forceinline__ int32_t pair_n_mma(int64_t N, int64_t n0) {
  const int64_t left = N - n0;
  return left >= BN ? BN : static_cast<int32_t>((left + 31) & ~int64_t{31});
}

template <int KIND, bool kSwiGLU, int BN>
__device__ __forceinline__ Tile get_pair_tile(const GParams& p, const GroupInfo& g, int64_t t, uint32_t crank) {
  const int64_t nt = (p.N + BN - 1) / BN;
  const int64_t mu = ((p.M + kBM - 1) / kBM + 1) / 2;
  Tile ti;
  ti.part = -1;
  ti.n_mma = BN;
  int64_t mp, nb;
  if (KIND == GEMM_GROUPED_M) {
    // Pair row tiles of 256 inside one expert, N-fastest; the odd CTA's half
    // of an expert's last tile may hold no rows of it (valid_m <= 0).
    const int32_t u = static_cast<int32_t>(t / nt);
    nb = t % nt;
    const int e = last_le(g.tile, p.n_groups, u);
    ti.m0 = static_cast<int64_t>(g.off[e]) + static_cast<int64_t>(u - g.tile[e]) * (2 * kBM) + crank * kBM;
    ti.a_row = ti.m0;
    if (kSwiGLU) {
      // Output features [128 nb, 128 nb + 128): the even CTA loads their gate
      // rows, the odd CTA their up rows (gate_up = [gate; up], N/2 rows each).
      ti.n0 = nb * (BN / 2);
      ti.b_row = static_cast<int64_t>(e) * p.b_rows_group + crank * (p.N >> 1) + ti.n0;
    } else {
      ti.n0 = nb * BN;
      ti.n_mma = pair_n_mma<BN>(p.N, ti.n0);
      ti.b_row = static_cast<int64_t>(e) * p.b_rows_group + ti.n0 + crank * (ti.n_mma / 2);
    }
    ti.k_atom0 = 0;
    ti.nkb = static_cast<int32_t>((p.K + kBK - 1) / kBK);
    ti.valid_m = static_cast<int32_t>(min64(kBM, g.off[e + 1] - ti.m0));  // >= -127
    ti.group = e;
    ti.sfb = p.b_scale;
    ti.cbase = p.c + ti.m0 * p.ldc + ti.n0;
    return ti;
  }
  if (KIND == GEMM_DENSE) {
    const int64_t nkb = (p.K + kBK - 1) / kBK;
    int64_t tt = t;
    ti.k_atom0 = 0;
    ti.nkb = static_cast<int32_t>(nkb);
    if (p.sk_w > 0 && t >= p.sk_first) {
      // Split tail: run `slot` is K blocks [slot*w, slot*w + w) of the tail
      // tiles laid end to end; segment 0 ends with its first tile, segment 1
      // is the remainder in the next tile.
      const int64_t v = t - p.sk_first;
      const int64_t slot = v % p.sk_slots, seg = v / p.sk_slots;
      const int64_t g0 = slot * p.sk_w, g1 = min64(g0 + p.sk_w, p.sk_total);
      const int64_t tile_end = (g0 / nkb + 1) * nkb;
      const int64_t lo = seg == 0 ? g0 : tile_end;
      const int64_t hi = seg == 0 ? min64(g1, tile_end) : g1;
      tt = p.sk_first;
      if (lo >= hi) {
        ti.part = -2;
        ti.nkb = 0;
      } else {
        const int64_t j = lo / nkb;
        tt = p.sk_first + j;
        ti.k_atom0 = lo - j * nkb;
        ti.nkb = static_cast<int32_t>(hi - lo);
        ti.part = static_cast<int32_t>(slot * 2 + seg);
      }
    }
    mp = p.n_fast ? tt / nt : tt % mu;
    nb = p.n_fast ? tt % nt : tt / mu;
    ti.group = 0;
  } else {
    const int64_t per = mu * nt;
    const int e = g.order[t / per];
    const int64_t rem = t % per;
    mp = rem % mu;
    nb = rem / mu;
    ti.k_atom0 = g.tile[e];
    ti.nkb = g.tile[e + 1] - g.tile[e];
    ti.group = e;
  }
  ti.m0 = (2 * mp + crank) * kBM;
  ti.n0 = nb * BN;
  ti.a_row = ti.m0;
  ti.n_mma = pair_n_mma<BN>(p.N, ti.n0);
  ti.b_row = ti.n0 + crank * (ti.n_mma / 2);
  ti.valid_m = static_cast<int32_t>(min64(kBM, p.M - ti.m0));
  ti.sfb = p.b_scale;
  ti.cbase = p.c + static_cast<int64_t>(ti.group) * p.c_group_stride + ti.m0 * p.ldc + ti.n0;
  return ti;
}

// Loads and checks the group offsets into shared memory; every thread calls.
// Returns false (after recording MX_ERR_DEVICE_CHECK) if they are invalid.
// tile_rows: rows of one M tile (rows-ragged prefix of tiles per expert).
template <int KIND>
__device__ bool setup_groups(const GParams& p, GroupInfo& g, int32_t* s_flag, int32_t* s_total,
                             int32_t tile_rows = 128) {
  const int tid = threadIdx.x;
  const int E = p.n_groups;
  if (tid == 0) *s_flag = 0;
  __syncthreads();
  const int64_t rows_total = (KIND == GEMM_GROUPED_M) ? p.M : -1;
  for (int e = tid; e <= E; e += blockDim.x) {
    const int64_t o = p.offsets[e];
    bool bad = (o < 0) || (o > 0x7FFFFFFFLL) || (e == 0 && o != 0);
    if (e == E && rows_total >= 0 && o != rows_total) bad = true;
    if (e > 0 && o < p.offsets[e - 1]) bad = true;
    g.off[e] = static_cast<int32_t>(o);
    if (bad) *s_flag = 1;
  }
  __syncthreads();
  if (*s_flag == 0) {
    if (tid == 0) {
      // Serial prefix: E <= 512 small integers, once per CTA.
      int32_t run = 0;
      int32_t prun = 0;
      for (int e = 0; e < E; ++e) {
        const int32_t m = g.off[e + 1] - g.off[e];
        g.tile[e] = run;
        run += (KIND == GEMM_GROUPED_M) ? (m + tile_rows - 1) / tile_rows : (m + 127) / 128;
        if (KIND == GEMM_GROUPED_M) {
          // rows-ragged: each expert's first column in a per-expert column copy
          // whose segments are padded to 128 rows (the SwiGLU epilogue's copy)
          g.order[e] = prun;
          prun += (m + 127) / 128 * 128;
        }
      }
      g.tile[E] = run;
      if (KIND == GEMM_GROUPED_M) {
        g.order[E] = prun;
        if (p.q_cap > 0 && prun > p.q_cap) *s_flag = 1;
      }
      *s_total = run;
      if (KIND == GEMM_GROUPED_K && static_cast<int64_t>(run) * 128 > p.K) *s_flag = 1;
    }
    __syncthreads();
    if (KIND == GEMM_GROUPED_K && *s_flag == 0) {
      // Experts ordered by decreasing K length (ties by index): rank sort.
      for (int e = tid; e < E; e += blockDim.x) {
        const int32_t me = g.tile[e + 1] - g.tile[e];
        int32_t rank = 0;
        for (int f = 0; f < E; ++f) {
          const int32_t mf = g.tile[f + 1] - g.tile[f];
          rank += (mf > me) || (mf == me && f < e);
        }
        g.order[rank] = e;
      }
    }
  }
  __syncthreads();
  g.total = *s_total;
  if (*s_flag != 0) {
    if (tid == 0 && blockIdx.x == 0 && p.dev_status) atomicExch(p.dev_status, static_cast<int>(MX_ERR_DEVICE_CHECK));
    return false;
  }
  return true;
}

__device__ __forceinline__ void record_timeout(const GParams& p, volatile int32_t* abort_flag) {
  *abort_flag = 1;
  if (p.dev_status) atomicExch(p.dev_status, static_cast<int>(MX_ERR_TIMEOUT));
}

// Bounded wait that also gives up once another role of the CTA has aborted.
// kCluster: acquire at cluster scope (barriers that the peer CTA signals).
template <bool kCluster = false>
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, const GParams& p,
                                              volatile int32_t* abort_flag) {
  auto test = [&]() { return kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
  if (test()) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (test()) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > p.timeout_ns) {
      record_timeout(p, abort_flag);
      return false;
    }
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Epilogue of the rows-ragged SwiGLU with its output quantised (the output's
// MX copies instead of the output): the values are rounded to BF16 exactly as
// the BF16 output would hold them, and coded as mx_quantize codes that output
// (both copies, per-expert column segments padded to 128 rows with zero codes).
// This thread holds row quarter * 32 + lane of the CTA's 128 rows and output
// features [n0 + 64 half, + 64) as FP32 in v[0 .. 63]; a warp's 32 rows are one
// 32-row block of the expert (tiles start at the expert's first row).
__device__ __forceinline__ void swiglu_quant_epilogue(const GParams& p, const QOut& q, const GroupInfo& g,
                                                      const Tile& ti, const uint32_t* v, int quarter, int half,
                                                      int lane, uint8_t* stg) {
  const int r = quarter * 32 + lane;
  const int64_t grow = ti.m0 + r;
  const bool rv = r < ti.valid_m;  // the row belongs to the tile's expert
  const int64_t f0 = ti.n0 + 64 * half;
  const int64_t F = p.n_out;
  const int64_t row_ka = (F + 127) / 128;
  const int64_t col_ka = (p.q_cap + 127) / 128;
  uint32_t w[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) w[j] = pack_bf16(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));

  // Row copy: the 1x32 blocks of features [f0, f0 + 32) and [f0 + 32, f0 + 64).
  // The warp's 32 rows x 64 codes are staged in its box (16-byte chunks
  // swizzled by row) and written back 8 rows x 64 contiguous bytes per store.
#pragma unroll
  for (int blk = 0; blk < 2; ++blk) {
    const uint32_t* wb = w + 16 * blk;
    uint32_t m = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) m = __vmaxu2(m, wb[j] & 0x7FFF7FFFu);
    const uint32_t code = scale_code(half_max(m));
    const bool nan_block = code == 0xFFu;
    const float inv = inv_scale(nan_block ? 0u : code);
    uint32_t c4[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      c4[j] = nan_block ? (nan_pair(wb[2 * j]) | (nan_pair(wb[2 * j + 1]) << 16)) : quant_quad(wb[2 * j], wb[2 * j + 1], inv);
    st_shared_v4(stg + lane * 64 + (((2 * blk) ^ (lane & 3)) << 4), make_uint4(c4[0], c4[1], c4[2], c4[3]));
    st_shared_v4(stg + lane * 64 + (((2 * blk + 1) ^ (lane & 3)) << 4), make_uint4(c4[4], c4[5], c4[6], c4[7]));
    if (rv) q.row_scale[scale_offset(grow, (f0 >> 5) + blk, row_ka)] = static_cast<uint8_t>(code);
  }
  __syncwarp();
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int rr = k * 8 + (lane >> 2);  // row of the warp's 32
    const int cc = lane & 3;             // 16-byte chunk of the row's 64 codes
    const uint4 c16 = ld_shared_v4(stg + rr * 64 + ((cc ^ (rr & 3)) << 4));
    if (quarter * 32 + rr < ti.valid_m)
      *reinterpret_cast<uint4*>(q.row_data + (ti.m0 + quarter * 32 + rr) * F + f0 + 16 * cc) = c16;
  }
  __syncwarp();  // the box is reused below

  // Column copy: per feature, the 32x1 block over this warp's rows; rows past
  // the expert's end are zero padding. A block wholly past the expert's
  // 128-padded segment belongs to no segment and is not written. The warp
  // transposes through its staging box, 32 features at a time: each lane
  // writes its row, then takes one feature's 32 values and codes them (its
  // block's amax, scale and 32 codes), one 32-byte store per feature.
  const int e = ti.group;
  const int64_t rel = ti.m0 - g.off[e] + quarter * 32;
  const int64_t seg = (static_cast<int64_t>(g.off[e + 1] - g.off[e]) + 127) / 128 * 128;
  if (rel < seg) {
    const int64_t cpos = g.order[e] + rel;  // column of the block's first row in the copy
    uint4* row_box = reinterpret_cast<uint4*>(stg + lane * 64);
    const uint16_t* col_box = reinterpret_cast<const uint16_t*>(stg);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const uint32_t* wh = w + 16 * hh;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        row_box[c] = rv ? make_uint4(wh[4 * c], wh[4 * c + 1], wh[4 * c + 2], wh[4 * c + 3]) : make_uint4(0u, 0u, 0u, 0u);
      __syncwarp();
      uint32_t x[16];  // the feature's 32 values, two per word (row 2k low, 2k + 1 high)
      uint32_t m = 0;
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        x[k] = static_cast<uint32_t>(col_box[(2 * k) * 32 + lane]) |
               (static_cast<uint32_t>(col_box[(2 * k + 1) * 32 + lane]) << 16);
        m = __vmaxu2(m, x[k] & 0x7FFF7FFFu);
      }
      __syncwarp();  // the box is rewritten by the next 32 features
      const uint32_t code = scale_code(half_max(m));
      const bool nan_block = code == 0xFFu;
      const float inv = inv_scale(nan_block ? 0u : code);
      uint32_t c4[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        c4[k] = nan_block ? (nan_pair(x[2 * k]) | (nan_pair(x[2 * k + 1]) << 16)) : quant_quad(x[2 * k], x[2 * k + 1], inv);
      const int64_t f = f0 + 32 * hh + lane;
      uint4* dst = reinterpret_cast<uint4*>(q.col_data + f * p.q_cap + cpos);
      dst[0] = make_uint4(c4[0], c4[1], c4[2], c4[3]);
      dst[1] = make_uint4(c4[4], c4[5], c4[6], c4[7]);
      q.col_scale[scale_offset(f, cpos >> 5, col_ka)] = static_cast<uint8_t>(code);
    }
  }
}

// Row-scale padding of the quantised SwiGLU output: rows [M, ceil(M/128)*128)
// belong to no expert; the first pair tile of each column tile (u == 0, even
// CTA) zeroes their four scale bytes of its 128 features, one row per
// epilogue thread.
__device__ __forceinline__ void swiglu_quant_row_padding(const GParams& p, const QOut& q, const Tile& ti,
                                                         int epi_thread) {
  const int64_t pad = (p.M + 127) / 128 * 128 - p.M;
  if (epi_thread < pad)
    *reinterpret_cast<uint32_t*>(q.row_scale + scale_offset(p.M + epi_thread, ti.n0 >> 5, (p.n_out + 127) / 128)) = 0u;
}

// Epilogue of one warp: its 32 rows (TMEM lane quarter) x my_chunks 32-column
// chunks starting at col_off, already in registers r[] (FP32 bit patterns).
template <int KIND, int kCols, int kBufs = 1>
__device__ __forceinline__ void store_tile(const GParams& p, const Tile& ti, const uint32_t* r, int quarter,
                                           int lane, int my_chunks, int col_off, uint8_t* stg,
                                           const CUtensorMap* tmap_c) {
  const int row = quarter * 32 + lane;
  if (MX_EPI_MODE == 1 && p.c_vec) {
    // Stage each 32-row x 32-column BF16 box in shared memory (64-byte
    // swizzle: conflict-free both ways) and write it back row-major, so one
    // warp store covers 8 rows x 64 contiguous bytes. Plain stores keep the
    // output off the TMA unit that streams the operands.
#pragma unroll
    for (int ch = 0; ch < kCols / 32; ++ch) {
      if (ch >= my_chunks) break;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int j = ch * 32 + q * 8;
        uint4 o;
        o.x = pack_bf16(__uint_as_float(r[j + 0]), __uint_as_float(r[j + 1]));
        o.y = pack_bf16(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
        o.z = pack_bf16(__uint_as_float(r[j + 4]), __uint_as_float(r[j + 5]));
        o.w = pack_bf16(__uint_as_float(r[j + 6]), __uint_as_float(r[j + 7]));
        st_shared_v4(stg + lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4), o);
      }
      __syncwarp();
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int rr = q * 8 + (lane >> 2);  // row within the box
        const int cc = lane & 3;             // 16-byte chunk within the row
        const uint4 v = ld_shared_v4(stg + rr * 64 + ((cc ^ ((rr >> 1) & 3)) << 4));
        const int trow = quarter * 32 + rr;
        const int64_t tcol = col_off + ch * 32 + cc * 8;
        const int64_t ncol = p.n_out - (ti.n0 + tcol);
        if (trow < ti.valid_m && ncol > 0) {
          __nv_bfloat16* dst = ti.cbase + static_cast<int64_t>(trow) * p.ldc + tcol;
          if (ncol >= 8) {
            *reinterpret_cast<uint4*>(dst) = v;
          } else {
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 8; ++e)
              if (e < ncol) reinterpret_cast<uint16_t*>(dst)[e] = static_cast<uint16_t>(w[e >> 1] >> ((e & 1) * 16));
          }
        }
      }
      __syncwarp();
    }
    return;
  }
  const bool tma_tile = p.c_tma && (KIND != GEMM_GROUPED_M || ti.valid_m == kBM);
  if (tma_tile) {
    // Stage 32-row x 32-column BF16 boxes in this warp's 64-byte-swizzled
    // buffer and let TMA write them (rows/columns outside C are clipped).
    const int32_t y = static_cast<int32_t>(ti.m0 + quarter * 32);
    const int32_t z = (KIND == GEMM_GROUPED_K) ? ti.group : 0;
#pragma unroll
    for (int ch = 0; ch < kCols / 32; ++ch) {
      if (ch >= my_chunks) break;
      // A staging box is free once its previous store has been read out;
      // with two boxes the most recent store may still be in flight.
      if (lane == 0) {
        if (kBufs == 2) bulk_wait_read_one_pending(); else bulk_wait_read_all();
      }
      __syncwarp();
      uint8_t* box = stg + (kBufs == 2 ? (ch & 1) * kEpiWarpBytes : 0);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int j = ch * 32 + q * 8;
        uint4 o;
        o.x = pack_bf16(__uint_as_float(r[j + 0]), __uint_as_float(r[j + 1]));
        o.y = pack_bf16(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
        o.z = pack_bf16(__uint_as_float(r[j + 4]), __uint_as_float(r[j + 5]));
        o.w = pack_bf16(__uint_as_float(r[j + 6]), __uint_as_float(r[j + 7]));
        st_shared_v4(box + lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4), o);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(tmap_c, box, static_cast<int32_t>(ti.n0 + col_off + ch * 32), y, z);
        bulk_commit_group();
      }
    }
  } else if (row < ti.valid_m) {
    const int64_t col0 = ti.n0 + col_off;
    const int64_t ncols = min64(my_chunks * 32, p.n_out - col0);
    __nv_bfloat16* dst = ti.cbase + static_cast<int64_t>(row) * p.ldc + col_off;
    if (ncols == my_chunks * 32 && p.c_vec) {
#pragma unroll
      for (int j = 0; j < kCols; j += 8) {
        if (j >= ncols) break;
        uint4 o;
        o.x = pack_bf16(__uint_as_float(r[j + 0]), __uint_as_float(r[j + 1]));
        o.y = pack_bf16(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
        o.z = pack_bf16(__uint_as_float(r[j + 4]), __uint_as_float(r[j + 5]));
        o.w = pack_bf16(__uint_as_float(r[j + 6]), __uint_as_float(r[j + 7]));
        *reinterpret_cast<uint4*>(dst + j) = o;
      }
    } else if (ncols > 0) {
#pragma unroll
      for (int j = 0; j < kCols; ++j)
        if (j < ncols) dst[j] = __float2bfloat16_rn(__uint_as_float(r[j]));
    }
  }
}

// ===========================================================================
// Single-CTA kernel (dense and grouped)
// ===========================================================================

template <int BN, int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                   const __grid_constant__ CUtensorMap tmap_c, const GParams p) {
  using C = Cfg<BN>;
  constexpr int S = C::kStages;
  constexpr int ACC = C::kAcc;
  constexpr bool kGatherSfa = (KIND == GEMM_GROUPED_M);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * C::kABytes;
  uint8_t* sSfa = sB + S * C::kBBytes;
  uint8_t* sSfb = sSfa + S * 512;
  uint8_t* sEpi = sSfb + S * C::kSfbBytes;  // 1024-aligned: the stage areas are multiples of 1024 bytes
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(sEpi + kEpiBytes);
  uint64_t* empty_bar = full_bar + S;
  uint64_t* acc_full = empty_bar + S;
  uint64_t* acc_empty = acc_full + ACC;
  uint64_t* drain_bar = acc_empty + ACC;
  uint64_t* sf_full = drain_bar + 1;
  uint64_t* sf_drain = sf_full + S;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sf_drain + 1);
  volatile int32_t* s_abort = reinterpret_cast<volatile int32_t*>(s_tmem + 1);
  int32_t* s_flag = reinterpret_cast<int32_t*>(s_tmem + 2);
  int32_t* s_total = reinterpret_cast<int32_t*>(s_tmem + 3);
  GroupInfo g;
  g.off = reinterpret_cast<int32_t*>(smem + C::smem_bytes(false) - 1024);
  g.tile = g.off + (kMaxGroups + 1);
  g.order = g.tile + (kMaxGroups + 1);
  g.total = 0;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Programmatic dependent launch: the next kernel on the stream may be
  // scheduled from here on; this grid touches global memory only after the
  // previous kernel has completed (grouped launches read the group offsets
  // first, dense launches wait after the on-chip setup).
  pdl_launch_dependents();
  if (KIND != GEMM_DENSE) {
    pdl_wait();
    if (!setup_groups<KIND>(p, g, s_flag, s_total)) return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      // Gathered scale atoms add one cp.async arrival per producer lane.
      mbar_init(&full_bar[s], kGatherSfa ? 33 : 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < ACC; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], kEpiThreads);
    }
    mbar_init(drain_bar, 1);
    for (int s = 0; s < S; ++s) mbar_init(&sf_full[s], 1);
    mbar_init(sf_drain, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (KIND == GEMM_DENSE) pdl_wait();
  const uint32_t tmem_base = *s_tmem;
  const int64_t ntiles = num_tiles<BN, KIND>(p, g);

  if (warp == 0) {
    // ------------------------------------------------------------- producer
    int stage = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    bool ok = true;
    // The whole warp only where it gathers scale words; otherwise lane 0 alone
    // (a per-stage warp shuffle slows the stage issue).
    for (int64_t t = blockIdx.x; t < ntiles && ok && (kGatherSfa || lane == 0); t += gridDim.x) {
      const Tile ti = get_tile<BN, KIND>(p, g, t);
      const int64_t sfb_row_atom0 = ti.n0 / 128;
      for (int kb = 0; kb < ti.nkb; ++kb) {
        const int64_t katom = ti.k_atom0 + kb;
        uint32_t good = 1;
        if (lane == 0) good = wait_or_abort(&empty_bar[stage], phase ^ 1, p, s_abort) ? 1u : 0u;
        if constexpr (kGatherSfa) good = __shfl_sync(0xFFFFFFFFu, good, 0);
        if (!good) {
          ok = false;
          break;
        }
        if constexpr (kGatherSfa) {
          // Scale bytes of A rows m0 .. m0+127 (any start row) gathered into one
          // atom with asynchronous 4-byte copies; each lane's arrival on the
          // stage's full barrier fires when its copies have landed, so the
          // producer never waits on them.
          uint8_t* dst = sSfa + stage * 512 + lane * 16;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int64_t r = ti.a_row + lane + 32 * q;
            const bool in = r < p.a_ra * 128;  // rows past the scale buffer read as zero
            cp_async_4(dst + 4 * q,
                       in ? p.a_scale + (((r >> 7) * p.ka + katom) << 9) + ((r & 31) << 4) + (((r >> 5) & 3) << 2)
                          : p.a_scale,
                       in ? 4u : 0u);
          }
          cp_async_arrive_noinc(&full_bar[stage]);
        }
        if (lane == 0) {
          uint32_t bytes = C::kABytes + C::kBBytes + (kGatherSfa ? 0 : 512);
#pragma unroll
          for (int j = 0; j < C::kSfbAtoms; ++j)
            if (sfb_row_atom0 + j < p.b_ra) bytes += 512;
          mbar_arrive_expect_tx(&full_bar[stage], bytes);
          const int32_t kx = static_cast<int32_t>(katom * kBK);
          tma_load_2d(sA + stage * C::kABytes, &tmap_a, &full_bar[stage], kx, static_cast<int32_t>(ti.a_row));
          tma_load_2d(sB + stage * C::kBBytes, &tmap_b, &full_bar[stage], kx, static_cast<int32_t>(ti.b_row));
          if constexpr (!kGatherSfa)
            bulk_load(sSfa + stage * 512, p.a_scale + (((ti.m0 >> 7) * p.ka + katom) << 9), 512, &full_bar[stage]);
#pragma unroll
          for (int j = 0; j < C::kSfbAtoms; ++j)
            if (sfb_row_atom0 + j < p.b_ra)
              bulk_load(sSfb + stage * C::kSfbBytes + j * 512, ti.sfb + (((sfb_row_atom0 + j) * p.ka + katom) << 9),
                        512, &full_bar[stage]);
        }
        ++issued;
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (*s_abort && lane == 0) {
      // Let the copies already issued land before the CTA goes away.
      int st = stage;
      uint32_t ph = phase;
      for (int64_t i = 0; i < min64(issued, S); ++i) {
        if (--st < 0) {
          st = S - 1;
          ph ^= 1;
        }
        mbar_wait(&full_bar[st], ph, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_mxf8_e4m3(kBM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const Tile ti = get_tile<BN, KIND>(p, g, t);
        if (!wait_or_abort(&acc_empty[acc], acc_phase ^ 1, p, s_abort)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < ti.nkb; ++kb) {
          // The copier issues a stage's scale copies only after its full
          // barrier completed, so the copies' barrier covers the operand tiles
          // as well: one wait per stage (a second one, on the full barrier,
          // cost ~50 cycles of every ~650-cycle stage).
          if (!wait_or_abort(&sf_full[stage], phase, p, s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t sfa_t = tmem_base + C::kSfCol0 + static_cast<uint32_t>(stage * C::kSfCols);
          const uint32_t sfb_t = sfa_t + 4;
          const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(sA + stage * C::kABytes));
          const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(sB + stage * C::kBBytes));
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            // +32 bytes along K inside the 128-byte swizzle atom = +2 in the address field.
            tc_mma_mxf8(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc_with_sf_id(idesc, k, k), sfa_t, sfb_t,
                        (kb | k) != 0 ? 1u : 0u);
          }
          tc_commit(&empty_bar[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(&acc_full[acc]);
        if (++acc == ACC) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      // All copies into and MMAs on tensor memory must finish before it is freed.
      tc_commit(drain_bar);
      mbar_wait(drain_bar, 0, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == kCopierWarp) {
    // -------------------------------------------------- scale-atom copier
    // A stage's scale slot in tensor memory is free again once the stage's
    // full barrier completes: the producer refilled the stage only after the
    // MMAs that read the slot's previous contents had committed.
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const Tile ti = get_tile<BN, KIND>(p, g, t);
        for (int kb = 0; kb < ti.nkb; ++kb) {
          if (!wait_or_abort(&full_bar[stage], phase, p, s_abort)) {
            ok = false;
            break;
          }
          // The gathered scale atom was written through the generic proxy; the
          // tensor-core copy reads it through the async proxy.
          if constexpr (kGatherSfa) fence_proxy_async_smem();
          tc_fence_after_sync();
          const uint32_t sfa = tmem_base + C::kSfCol0 + static_cast<uint32_t>(stage * C::kSfCols);
          tc_cp_32x128b_warpx4(sfa, sdesc_scale_atom(smem_u32(sSfa + stage * 512)));
#pragma unroll
          for (int j = 0; j < C::kSfbAtoms; ++j)
            tc_cp_32x128b_warpx4(sfa + 4 + 4 * j, sdesc_scale_atom(smem_u32(sSfb + stage * C::kSfbBytes + j * 512)));
          tc_commit(&sf_full[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      tc_commit(sf_drain);
      mbar_wait(sf_drain, 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- epilogue
    const int quarter = warp & 3;         // TMEM lanes this warp may read
    const int half = (warp - 2) >> 2;     // which part of the tile's columns
    constexpr int kChunks = BN / 32;      // 32-column chunks of the tile
    constexpr int kHalf0 = (kChunks + 1) / 2;
    constexpr int kCols = kHalf0 * 32;    // register columns per thread
    const int my_chunks = half == 0 ? kHalf0 : kChunks - kHalf0;
    const int col_off = half * kHalf0 * 32;
    uint8_t* stg = sEpi + (warp - 2) * kEpiWarpBytes;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
      const Tile ti = get_tile<BN, KIND>(p, g, t);
      if (!wait_or_abort(&acc_full[acc], acc_phase, p, s_abort)) break;
      tc_fence_after_sync();
      uint32_t r[kCols];
      if (ti.nkb > 0) {
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                               static_cast<uint32_t>(acc * BN + col_off);
#pragma unroll
        for (int ch = 0; ch < kHalf0; ++ch)
          if (ch < my_chunks) tmem_ld_32x32b_x32(taddr + ch * 32, r + ch * 32);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int i = 0; i < kCols; ++i) r[i] = 0u;  // empty contraction: exact zeros
      }
      tc_fence_before_sync();
      mbar_arrive(&acc_empty[acc]);
      if (++acc == ACC) {
        acc = 0;
        acc_phase ^= 1;
      }
      store_tile<KIND, kCols>(p, ti, r, quarter, lane, my_chunks, col_off, stg, &tmap_c);
    }
    // Bulk stores must have completed before the CTA's shared memory goes away.
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ===========================================================================
// CTA-pair kernel (dense and both grouped kinds): clusters of two, tcgen05
// cta_group::2, M = 256
// ===========================================================================

// Parameters of one pair-kernel launch: up to kMaxProblems independent dense
// GEMMs whose tiles one persistent grid walks in turn (problem i owns launch
// tiles [tile0[i], tile0[i+1])), or a single GEMM of any kind (n = 1).
constexpr int kMaxProblems = MX_MAX_GEMM_MULTI;
// A balanced schedule (sched = 1) gives cluster c cnt[i][c] consecutive tiles
// of problem i, starting after the tiles of clusters 0 .. c-1; otherwise
// cluster c takes launch tiles c, c + clusters, ... .
constexpr int kMaxSchedClusters = 96;
struct PairProblem {
  CUtensorMap a, b, sfa, sfb, c;
  GParams p;
};
struct PairArgs {
  PairProblem prob[kMaxProblems];
  int64_t tile0[kMaxProblems + 1];
  QOut q;  // the quantised SwiGLU epilogue's outputs (single problem)
  int n;
  int sched;
  uint8_t cnt[kMaxProblems][kMaxSchedClusters];
};
static_assert(sizeof(PairArgs) <= 4096, "kernel parameter space");

template <bool kMulti>
__device__ __forceinline__ int problem_of(const PairArgs& args, int64_t t) {
  int i = 0;
  if constexpr (kMulti)
    while (i + 1 < args.n && t >= args.tile0[i + 1]) ++i;
  return i;
}

// kSwiGLU_: 0 none; 1 the SwiGLU epilogue writes its BF16 output; 2 it writes
// the output's MX copies instead.
template <int KIND, int kSwiGLU_, bool kMulti, int BN_, bool kTS>
__global__ void __launch_bounds__(kPairThreads, 1)
    mx_gemm_pair_kernel(const __grid_constant__ PairArgs args) {
  constexpr bool kSwiGLU = kSwiGLU_ != 0;
  constexpr bool kSwiQ = kSwiGLU_ == 2;
  using C = PairCfgT<BN_, kTS, KIND != GEMM_DENSE>;
  static_assert(!kMulti || (KIND == GEMM_DENSE && !kSwiGLU), "several problems per launch: dense GEMMs only");
  // Problem 0 holds the fields every problem shares (status word, wait bound)
  // and, unless kMulti, the whole GEMM.
  const GParams& p = args.prob[0].p;
  static_assert(!kSwiGLU || (KIND == GEMM_GROUPED_M && BN_ == 256 && !kTS),
                "the SwiGLU epilogue follows the grouped gate_up fprop");
  // Rows-ragged tiles start at any row: each CTA gathers its A scale atom.
  constexpr bool kGatherSfa = (KIND == GEMM_GROUPED_M) && !kTS;
  constexpr bool kGather = kGatherSfa;
  constexpr int S = C::kStages;
  constexpr int BN = C::BN;
  constexpr int ACC = C::kAcc;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // Operand tiles (1024-byte aligned for the 128-byte swizzle), the epilogue's
  // staging boxes (1024-byte aligned), then the scale atoms (16-byte aligned).
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * C::kABytes;
  uint8_t* sEpi = sB + S * C::kBBytes;
  uint8_t* sSfa = sEpi + C::kEpiBufs * kEpiBytes;
  uint8_t* sSfb = sSfa + S * C::kSfaBytes;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(sSfb + S * C::kSfbBytes);  // used in the even CTA
  uint64_t* empty_bar = full_bar + S;
  uint64_t* acc_full = empty_bar + S;  // [ACC]
  uint64_t* acc_empty = acc_full + 2;  // [ACC], used in the even CTA
  uint64_t* drain_bar = acc_empty + 2;
  uint64_t* sf_full = drain_bar + 1;  // used in the even CTA
  uint64_t* sf_drain = sf_full + S;
  uint64_t* gfull = sf_drain + 1;  // odd CTA: its own gathered scale atom landed
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(gfull + S);
  volatile int32_t* s_abort = reinterpret_cast<volatile int32_t*>(s_tmem + 1);
  int32_t* s_flag = reinterpret_cast<int32_t*>(s_tmem + 2);
  int32_t* s_total = reinterpret_cast<int32_t*>(s_tmem + 3);
  int32_t* s_seq = reinterpret_cast<int32_t*>(s_tmem + 4);  // scheduled: [first tile of each problem][count]
  GroupInfo g;
  g.off = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(s_tmem) + 16 + 2 * MX_MAX_GEMM_MULTI * 4);
  g.tile = g.off + (kMaxGroups + 1);
  g.order = g.tile + (kMaxGroups + 1);
  g.total = 0;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const bool leader = crank == 0;

  // Programmatic dependent launch, as in mx_gemm_kernel. Both CTAs of a pair
  // read the same offsets and reach the same verdict.
  pdl_launch_dependents();
  if (KIND != GEMM_DENSE) {
    pdl_wait();
    if (!setup_groups<KIND>(p, g, s_flag, s_total, 2 * kBM)) return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      // The leader's expect_tx (both CTAs' loads complete the bytes); with a
      // scale gather also the leader's 32 cp.async lanes and the odd CTA's relay.
      mbar_init(&full_bar[s], kGather ? 34 : 1);
      mbar_init(&empty_bar[s], 1);  // the leader's MMA commit, multicast to both CTAs
      mbar_init(&gfull[s], 32);
    }
    for (int a = 0; a < ACC; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 16);  // one arrival per epilogue warp of both CTAs
    }
    mbar_init(drain_bar, 1);
    for (int s = 0; s < S; ++s) mbar_init(&sf_full[s], 1);
    mbar_init(sf_drain, 1);
    *s_abort = 0;
    if (kMulti && args.sched) {
      // This cluster's range of each problem's tiles.
      const int c = static_cast<int>(blockIdx.x >> 1);
      for (int i = 0; i < args.n; ++i) {
        int32_t first = 0;
        for (int q = 0; q < c; ++q) first += args.cnt[i][q];
        s_seq[i] = first;
        s_seq[kMaxProblems + i] = args.cnt[i][c];
      }
    }
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < (kMulti ? args.n : 1); ++i) {
      tma_prefetch_desc(&args.prob[i].a);
      tma_prefetch_desc(&args.prob[i].b);
      if (!kTS && !kGatherSfa) tma_prefetch_desc(&args.prob[i].sfa);
      if (!kTS) tma_prefetch_desc(&args.prob[i].sfb);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(s_tmem, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();  // barriers of both CTAs exist before either signals the other
  tc_fence_after_sync();
  if (KIND == GEMM_DENSE) pdl_wait();
  const uint32_t tmem_base = *s_tmem;
  const int64_t nt = (p.N + BN - 1) / BN;
  int64_t ntiles = (KIND == GEMM_GROUPED_M)
                       ? static_cast<int64_t>(g.total) * nt
                       : (((p.M + kBM - 1) / kBM + 1) / 2) * nt * (KIND == GEMM_GROUPED_K ? p.n_groups : 1);
  if (KIND == GEMM_DENSE && p.sk_w > 0) ntiles = p.sk_first + 2 * static_cast<int64_t>(p.sk_slots);
  if (kMulti) ntiles = args.tile0[args.n];
  const int64_t t_first = blockIdx.x >> 1;
  const int64_t t_step = gridDim.x >> 1;
  // The i-th launch tile of this cluster, or -1 past its last.
  const bool sched = kMulti && args.sched;
  auto next_tile = [&](int64_t i) -> int64_t {
    if (!sched) {
      const int64_t t = t_first + i * t_step;
      return t < ntiles ? t : -1;
    }
    for (int q = 0; q < args.n; ++q) {
      const int64_t cnt = s_seq[kMaxProblems + q];
      if (i < cnt) return args.tile0[q] + s_seq[q] + i;
      i -= cnt;
    }
    return -1;
  };

  if (warp == 0) {
    // ------------------------------------------------------------- producer
    int stage = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    bool ok = true;
    // Lane 0 alone runs the loop (the rows-ragged scale gather has a warp of
    // its own: a per-stage warp shuffle here cost ~5% of GEMM throughput).
    for (int64_t it = 0, t; lane == 0 && ok && (t = next_tile(it)) >= 0; ++it) {
      const int pi = problem_of<kMulti>(args, t);
        const GParams& pp = args.prob[pi].p;
        const Tile ti = get_pair_tile<KIND, kSwiGLU, BN>(pp, g, kMulti ? t - args.tile0[pi] : t, crank);
      // Rows-ragged: B's scale atoms are those of the tile's expert. SwiGLU:
      // the second atom holds the up rows, N/256 atoms after the gate rows.
      const int64_t sfb_atom_row = (KIND == GEMM_GROUPED_M ? ti.group * pp.b_ra : 0) + (ti.n0 >> 7);
      const int64_t sfb_atom_step = kSwiGLU ? (pp.N >> 8) : 1;
      for (int kb = 0; kb < ti.nkb; ++kb) {
        if (!wait_or_abort<true>(&empty_bar[stage], phase ^ 1, p, s_abort)) {
          ok = false;
          break;
        }
        const int64_t katom = ti.k_atom0 + kb;
        {
          const uint32_t lfull = mapa_shared(smem_u32(&full_bar[stage]), 0);
          // Both CTAs' TMA bytes complete on the leader's barrier; gathered
          // scale words arrive through the gather warps instead.
          if (leader)
            mbar_arrive_expect_tx(&full_bar[stage], 2 * (C::kStageTx - (kGatherSfa ? C::kSfaBytes : 0)));
          const int32_t kx = static_cast<int32_t>(katom * kBK);
          tma_load_2d_pair(sA + stage * C::kABytes, &args.prob[pi].a, lfull, kx, static_cast<int32_t>(ti.a_row));
          tma_load_2d_pair(sB + stage * C::kBBytes, &args.prob[pi].b, lfull, kx, static_cast<int32_t>(ti.b_row));
          // Scale atoms through [atoms][128 words] views (rows past the end read as zero).
          if constexpr (!kTS && !kGatherSfa)
            tma_load_2d_pair(sSfa + stage * C::kSfaBytes, &args.prob[pi].sfa, lfull, 0,
                             static_cast<int32_t>((ti.m0 >> 7) * pp.ka + katom));
          if constexpr (!kTS) {
#pragma unroll
            for (int j = 0; j < 2; ++j)
              tma_load_2d_pair(sSfb + stage * C::kSfbBytes + j * 512, &args.prob[pi].sfb, lfull, 0,
                               static_cast<int32_t>((sfb_atom_row + j * sfb_atom_step) * pp.ka + katom));
          }
        }
        ++issued;
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (*s_abort && leader && lane == 0) {
      // The leader's full barriers count both CTAs' copies: let them land.
      int st = stage;
      uint32_t ph = phase;
      for (int64_t i = 0; i < min64(issued, S); ++i) {
        if (--st < 0) {
          st = S - 1;
          ph ^= 1;
        }
        mbar_wait(&full_bar[st], ph, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------- MMA issuer (even CTA)
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = kTS ? idesc_f8_e4m3_f32(2 * kBM, BN) : idesc_mxf8_e4m3(2 * kBM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int64_t it = 0, t; ok && (t = next_tile(it)) >= 0; ++it) {
        const int pi = problem_of<kMulti>(args, t);
        const GParams& pp = args.prob[pi].p;
        const Tile ti = get_pair_tile<KIND, kSwiGLU, BN>(pp, g, kMulti ? t - args.tile0[pi] : t, crank);
        if (ti.part == -2) continue;  // an empty split-tail segment
        if (!wait_or_abort<true>(&acc_empty[acc], acc_phase ^ 1, p, s_abort)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        const uint32_t idesc_t = ti.n_mma == BN ? idesc
                                 : (kTS ? idesc_f8_e4m3_f32(2 * kBM, static_cast<uint32_t>(ti.n_mma))
                                        : idesc_mxf8_e4m3(2 * kBM, static_cast<uint32_t>(ti.n_mma)));
        for (int kb = 0; kb < ti.nkb; ++kb) {
          // With block scales the copier's barrier covers the operand tiles
          // too (it copies a stage's scales only after the stage's full
          // barrier, which counts both CTAs' loads, completed), so the issuer
          // waits once per stage, on its own CTA's barrier.
          if (!(kTS ? wait_or_abort<true>(&full_bar[stage], phase, p, s_abort)
                    : wait_or_abort<false>(&sf_full[stage], phase, p, s_abort))) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(sA + stage * C::kABytes));
          const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(sB + stage * C::kBBytes));
          if constexpr (kTS) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc_mma_f8_pair(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc_t, (kb | k) != 0 ? 1u : 0u);
          } else {
            const uint32_t sfa_t = tmem_base + C::kSfCol0 + static_cast<uint32_t>(stage * C::kSfCols);
            const uint32_t sfb_t = sfa_t + 4;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc_mma_mxf8_pair(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc_with_sf_id(idesc_t, k, k), sfa_t, sfb_t,
                               (kb | k) != 0 ? 1u : 0u);
          }
          tc_commit_pair_multicast(&empty_bar[stage], static_cast<uint16_t>(0x3));
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit_pair_multicast(&acc_full[acc], static_cast<uint16_t>(0x3));
        if (++acc == ACC) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      // All copies into and MMAs on tensor memory must finish before it is freed.
      tc_commit_pair_multicast(drain_bar, static_cast<uint16_t>(0x1));
      mbar_wait(drain_bar, 0, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == kCopierWarp) {
    // ------------------------------------- scale-atom copier (even CTA)
    // A stage's slot in tensor memory is free again once its full barrier
    // completes: the producer refilled the stage only after the MMAs that
    // read the previous contents had committed.
    if (lane == 0 && !leader && kGather) {
      // Odd CTA: forward each stage's landed scale gather to the leader's full
      // barrier, after making it visible to the tensor-core copies. The words
      // sit in this CTA's own shared memory and are read by this SM's share of
      // the pair-wide copy, which the leader can only issue after seeing this
      // arrival; a CTA-scope arrive therefore suffices (a cluster-scope release
      // here cost a third of the kernel's throughput).
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int64_t it = 0, t; ok && (t = next_tile(it)) >= 0; ++it) {
        const int pi = problem_of<kMulti>(args, t);
        const GParams& pp = args.prob[pi].p;
        const Tile ti = get_pair_tile<KIND, kSwiGLU, BN>(pp, g, kMulti ? t - args.tile0[pi] : t, crank);
        for (int kb = 0; kb < ti.nkb; ++kb) {
          if (!wait_or_abort(&gfull[stage], phase, p, s_abort)) {
            ok = false;
            break;
          }
          fence_proxy_async_smem();
          mbar_arrive_cluster(mapa_shared(smem_u32(&full_bar[stage]), 0));
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
    if (lane == 0 && leader && !kTS) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int64_t it = 0, t; ok && (t = next_tile(it)) >= 0; ++it) {
        const int pi = problem_of<kMulti>(args, t);
        const GParams& pp = args.prob[pi].p;
        const Tile ti = get_pair_tile<KIND, kSwiGLU, BN>(pp, g, kMulti ? t - args.tile0[pi] : t, crank);
        for (int kb = 0; kb < ti.nkb; ++kb) {
          if (!wait_or_abort<true>(&full_bar[stage], phase, p, s_abort)) {
            ok = false;
            break;
          }
          // The leader's gathered words were written through the generic proxy.
          if constexpr (kGather) fence_proxy_async_smem();
          tc_fence_after_sync();
          const uint32_t sfa = tmem_base + C::kSfCol0 + static_cast<uint32_t>(stage * C::kSfCols);
          tc_cp_32x128b_warpx4_pair(sfa, sdesc_scale_atom(smem_u32(sSfa + stage * C::kSfaBytes)));
          tc_cp_32x128b_warpx4_pair(sfa + 4, sdesc_scale_atom(smem_u32(sSfb + stage * C::kSfbBytes)));
          tc_cp_32x128b_warpx4_pair(sfa + 8, sdesc_scale_atom(smem_u32(sSfb + stage * C::kSfbBytes + 512)));
          tc_commit_pair_multicast(&sf_full[stage], static_cast<uint16_t>(0x1));
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      tc_commit_pair_multicast(sf_drain, static_cast<uint16_t>(0x1));
      mbar_wait(sf_drain, 0, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == kGatherWarp) {
    // ----------------------------------------- A scale gather (rows-ragged)
    // Scale words of A rows m0 .. m0+127 (any start row) gathered into the
    // stage's atom with 4-byte asynchronous copies; each lane's arrival fires
    // when its copies have landed (the leader's full barrier, or the odd
    // CTA's local barrier that its relay warp forwards to the leader).
    if constexpr (kGather) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int64_t it = 0, t; ok && (t = next_tile(it)) >= 0; ++it) {
        const int pi = problem_of<kMulti>(args, t);
        const GParams& pp = args.prob[pi].p;
        const Tile ti = get_pair_tile<KIND, kSwiGLU, BN>(pp, g, kMulti ? t - args.tile0[pi] : t, crank);
        for (int kb = 0; kb < ti.nkb; ++kb) {
          uint32_t good = 1;
          if (lane == 0) good = wait_or_abort<true>(&empty_bar[stage], phase ^ 1, p, s_abort) ? 1u : 0u;
          good = __shfl_sync(0xFFFFFFFFu, good, 0);
          if (!good) {
            ok = false;
            break;
          }
          const int64_t katom = ti.k_atom0 + kb;
          if constexpr (kGatherSfa) {
            uint8_t* dst = sSfa + stage * C::kSfaBytes + lane * 16;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int64_t r = ti.a_row + lane + 32 * q;
              const bool in = r < pp.a_ra * 128;  // rows past the scale buffer read as zero
              cp_async_4(dst + 4 * q,
                         in ? pp.a_scale + (((r >> 7) * pp.ka + katom) << 9) + ((r & 31) << 4) + (((r >> 5) & 3) << 2)
                            : pp.a_scale,
                         in ? 4u : 0u);
            }
          }
          cp_async_arrive_noinc(leader ? &full_bar[stage] : &gfull[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      cp_async_wait_all();  // no copy into this CTA's memory outlives it
    }
    __syncwarp();
  } else {
    // ------------------------------------------------- epilogue (both CTAs)
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    constexpr int kCols = BN / 2;
    const int col_off = half * kCols;
    uint8_t* stg = sEpi + (warp - 2) * C::kEpiBufs * kEpiWarpBytes;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int64_t it = 0, t; (t = next_tile(it)) >= 0; ++it) {
      const int pi = problem_of<kMulti>(args, t);
      const GParams& pp = args.prob[pi].p;
      const Tile ti = get_pair_tile<KIND, kSwiGLU, BN>(pp, g, kMulti ? t - args.tile0[pi] : t, crank);
      if (ti.part == -2) continue;
      float ts = 1.0f;  // the tile's product of tensor scales (kTS), read while the MMAs run
      if constexpr (kTS) ts = __ldg(pp.ts_a) * __ldg(pp.ts_b + (KIND == GEMM_GROUPED_M ? ti.group : 0));
      if (!wait_or_abort<true>(&acc_full[acc], acc_phase, p, s_abort)) break;
      tc_fence_after_sync();
      uint32_t r[kCols];
      if (ti.nkb > 0) {
        if (kSwiGLU) {
          // Features [64 half, 64 half + 64): gate columns then the up columns
          // 128 further on.
          const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(64 * half);
          tmem_ld_32x32b_x32(taddr, r);
          tmem_ld_32x32b_x32(taddr + 32, r + 32);
          tmem_ld_32x32b_x32(taddr + 128, r + 64);
          tmem_ld_32x32b_x32(taddr + 160, r + 96);
        } else {
          const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                 static_cast<uint32_t>(acc * BN + col_off);
#pragma unroll
          for (int ch = 0; ch < kCols / 32; ++ch) tmem_ld_32x32b_x32(taddr + ch * 32, r + ch * 32);
        }
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int i = 0; i < kCols; ++i) r[i] = 0u;
      }
      tc_fence_before_sync();
      __syncwarp();
      // the even CTA's MMAs may overwrite this accumulator
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&acc_empty[acc]), 0));
      if (++acc == ACC) {
        acc = 0;
        acc_phase ^= 1;
      }
      if constexpr (kTS) {
#pragma unroll
        for (int i = 0; i < kCols; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * ts);
      }
      if constexpr (KIND == GEMM_DENSE && BN == 256 && !kTS) {
        if (ti.part >= 0) {
          // Split-tail segment: the FP32 partial goes to the workspace.
          float4* dst = reinterpret_cast<float4*>(pp.ws) +
                        ((static_cast<int64_t>(ti.part) * 2 + crank) * 8 + (warp - 2)) * (32 * 32) + lane;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            dst[j * 32] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                      __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
          continue;
        }
      }
      if constexpr (kSwiGLU) {
        // SwiGLU in FP32 on the FP32 accumulators, one rounding to BF16 at the store
        // (the fast exponential's error stays below 1e-5 relative for |x| < 88).
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const float gv = __uint_as_float(r[i]);
          const float uv = __uint_as_float(r[64 + i]);
          r[i] = __float_as_uint(gv / (1.0f + __expf(-gv)) * uv);
        }
        if constexpr (kSwiQ) {
          swiglu_quant_epilogue(pp, args.q, g, ti, r, quarter, half, lane, stg);
          if (crank == 0 && t < nt) swiglu_quant_row_padding(pp, args.q, ti, (warp - 2) * 32 + lane);
        } else {
          store_tile<KIND, 64, C::kEpiBufs>(pp, ti, r, quarter, lane, 2, 64 * half, stg, &args.prob[pi].c);
        }
      } else {
        store_tile<KIND, kCols, C::kEpiBufs>(pp, ti, r, quarter, lane, kCols / 32, col_off, stg, &args.prob[pi].c);
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the other may still signal it
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// ===========================================================================
// Split-tail reduction
// ===========================================================================
//
// Tail tile j's FP32 partials, one per run of K blocks that touched it, are
// added in run order (so repeated calls give identical bits) and rounded to
// BF16 once, as the GEMM epilogue does. Block (2j + r) * 16 + c handles the
// r-th CTA's 128 rows and the 8-column chunk c of each epilogue warp's half:
// thread (w, lane) holds row `lane` of epilogue warp w + 2, so its partials
// are two float4 of every unit, and the loads of up to four units are in
// flight at once.
__global__ void __launch_bounds__(256) mx_gemm_sk_reduce_kernel(const GParams p) {
  // The partials come from the GEMM launch before this one; the next kernel is
  // let in once this CTA's stores are issued (as in the blockwise GEMM).
  pdl_wait();
  const int64_t nkb = (p.K + kBK - 1) / kBK;
  const int c = blockIdx.x & 15;
  const int crank = (blockIdx.x >> 4) & 1;
  const int64_t j = blockIdx.x >> 5;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = (w + 2) & 3, half = w >> 2;
  const int64_t nt = (p.N + PairCfg::BN - 1) / PairCfg::BN;
  const int64_t mu = ((p.M + kBM - 1) / kBM + 1) / 2;
  const int64_t tt = p.sk_first + j;
  const int64_t mp = p.n_fast ? tt / nt : tt % mu;
  const int64_t nb = p.n_fast ? tt % nt : tt / mu;
  const int64_t row = (2 * mp + crank) * kBM + quarter * 32 + lane;
  const int64_t col = nb * PairCfg::BN + half * 128 + 8 * c;
  const int64_t s_lo = j * nkb / p.sk_w, s_hi = ((j + 1) * nkb - 1) / p.sk_w;
  const float4* base = reinterpret_cast<const float4*>(p.ws) + (crank * 8 + w) * (32 * 32) + (2 * c) * 32 + lane;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  for (int64_t s0 = s_lo; s0 <= s_hi; s0 += 4) {
    float4 v[4][2];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t slot = s0 + u;
      if (slot <= s_hi) {
        const int64_t unit = slot * 2 + (slot * p.sk_w >= j * nkb ? 0 : 1);
        const float4* src = base + unit * (kPartialFloats / 4);
        v[u][0] = __ldcs(src);
        v[u][1] = __ldcs(src + 32);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (s0 + u <= s_hi) {  // in run order
        acc[0] += v[u][0].x;
        acc[1] += v[u][0].y;
        acc[2] += v[u][0].z;
        acc[3] += v[u][0].w;
        acc[4] += v[u][1].x;
        acc[5] += v[u][1].y;
        acc[6] += v[u][1].z;
        acc[7] += v[u][1].w;
      }
    }
  }
  if (row < p.M && col < p.n_out) {
    __nv_bfloat16* dst = p.c + row * p.ldc + col;
    const uint32_t wv[4] = {pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]), pack_bf16(acc[4], acc[5]),
                            pack_bf16(acc[6], acc[7])};
    if (p.c_vec && col + 8 <= p.n_out) {
      *reinterpret_cast<uint4*>(dst) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (col + e < p.n_out) reinterpret_cast<uint16_t*>(dst)[e] = static_cast<uint16_t>(wv[e >> 1] >> ((e & 1) * 16));
    }
  }
  pdl_launch_dependents();
}

// ===========================================================================
// Blockwise FP8 variant (DeepSeek-V3 recipe): C = sum over 128-K blocks of
// (A_kb . B_kb^T) / (s_a[kb][m] * s_b[n/128][kb])
// ===========================================================================
//
// "浮点格式、数值稳定性与混合精度" §七.3: the block scales change along K, so
// each 128-K block's partial sum is promoted to FP32 with its two scales. Here
// the tensor core computes each block's partial sum (plain E4M3 MMAs, exact
// products, FP32 accumulation, no block scales) into one of two TMEM buffers,
// and the epilogue warps fold it into FP32 registers while the MMAs fill the
// other buffer. 128 x 256 tiles: the two 256-column partial buffers take all
// of TMEM (no scale columns are needed); 128 x 128 tiles for narrow outputs.

template <int BN_>
struct BwCfg {
  static constexpr int BN = BN_;
  static constexpr int kStages = BN == 256 ? 4 : 6;
  // Epilogue warps: four per TMEM lane quarter at BN = 256 (64 columns each),
  // two at BN = 128.
  static constexpr int kEpiWarps = BN == 256 ? 16 : 8;
  static constexpr int kThreads = (2 + kEpiWarps) * 32;
  static constexpr int kEpiStage = kEpiWarps * kEpiWarpBytes;
  static constexpr int kParts = 2;  // partial-sum buffers in TMEM (a third measured no faster)
  static constexpr int kABytes = kBM * kBK;
  static constexpr int kBBytes = BN * kBK;
  static_assert(kParts * BN <= kTmemCols, "TMEM budget");
  static constexpr int kBarBytes = (2 * kStages + 2 * kParts + 1) * 8 + 16;
  static constexpr size_t smem_bytes() {
    return 1024 + static_cast<size_t>(kStages) * (kABytes + kBBytes) + kEpiStage + kBarBytes;
  }
};

template <int BN_>
__global__ void __launch_bounds__(BwCfg<BN_>::kThreads, 1)
    mx_gemm_blockwise_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                             const __grid_constant__ CUtensorMap tmap_c, const GParams p,
                             const float* __restrict__ sa, const float* __restrict__ sb) {
  using C = BwCfg<BN_>;
  constexpr int S = C::kStages;
  constexpr int BN = C::BN;
  constexpr int kSplit = C::kEpiWarps / 4;  // epilogue warps sharing a TMEM lane quarter
  constexpr int kCols = BN / kSplit;       // columns per epilogue thread (its TMEM lane)

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * C::kABytes;
  uint8_t* sEpi = sB + S * C::kBBytes;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(sEpi + C::kEpiStage);
  uint64_t* empty_bar = full_bar + S;
  constexpr int P = C::kParts;
  uint64_t* part_full = empty_bar + S;   // [P] a partial sum is in TMEM
  uint64_t* part_empty = part_full + P;  // [P] the epilogue has read it
  uint64_t* drain_bar = part_empty + P;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int32_t* s_abort = reinterpret_cast<volatile int32_t*>(s_tmem + 1);
  GroupInfo g{};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < P; ++b) {
      mbar_init(&part_full[b], 1);
      mbar_init(&part_empty[b], C::kEpiWarps * 32);
    }
    mbar_init(drain_bar, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  // Programmatic dependent launch: global memory only once the previous
  // kernel on the stream has completed. The next kernel is let in only after
  // this CTA's tiles (below): the registers and shared memory this kernel
  // leaves free hold a small CTA, and one waiting there would take issue
  // slots from the promotion.
  pdl_wait();
  const uint32_t tmem_base = *s_tmem;
  const int64_t ntiles = ((p.M + kBM - 1) / kBM) * ((p.N + BN - 1) / BN);
  const int64_t kbs = (p.K + kBK - 1) / kBK;
  const int64_t nbw = (p.N + 127) / 128;  // weight blocks along N

  if (warp == 0) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const Tile ti = get_tile<BN, GEMM_DENSE>(p, g, t);
        for (int kb = 0; kb < ti.nkb; ++kb) {
          if (!wait_or_abort(&empty_bar[stage], phase ^ 1, p, s_abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full_bar[stage], C::kABytes + C::kBBytes);
          const int32_t kx = kb * kBK;
          tma_load_2d(sA + stage * C::kABytes, &tmap_a, &full_bar[stage], kx, static_cast<int32_t>(ti.a_row));
          tma_load_2d(sB + stage * C::kBBytes, &tmap_b, &full_bar[stage], kx, static_cast<int32_t>(ti.b_row));
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (*s_abort) {
        int st = stage;
        uint32_t ph = phase;
        for (int64_t i = 0; i < min64(issued, S); ++i) {
          if (--st < 0) {
            st = S - 1;
            ph ^= 1;
          }
          mbar_wait(&full_bar[st], ph, p.timeout_ns);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f8_e4m3_f32(kBM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int64_t gk = 0;  // k blocks issued so far: buffer gk % P, its use count gk / P
      bool ok = true;
      for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const Tile ti = get_tile<BN, GEMM_DENSE>(p, g, t);
        for (int kb = 0; kb < ti.nkb; ++kb, ++gk) {
          const int buf = static_cast<int>(gk % P);
          if (!wait_or_abort(&full_bar[stage], phase, p, s_abort) ||
              !wait_or_abort(&part_empty[buf], static_cast<uint32_t>(((gk / P) & 1) ^ 1), p, s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
          const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(sA + stage * C::kABytes));
          const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(sB + stage * C::kBBytes));
#pragma unroll
          for (int k = 0; k < 4; ++k) tc_mma_f8(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, k != 0 ? 1u : 0u);
          tc_commit(&empty_bar[stage]);
          tc_commit(&part_full[buf]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      tc_commit(drain_bar);
      mbar_wait(drain_bar, 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int part = (warp - 2) >> 2;  // which kCols-wide slice of the tile
    const int col_off = part * kCols;
    uint8_t* stg = sEpi + (warp - 2) * kEpiWarpBytes;
    int64_t gk = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
      const Tile ti = get_tile<BN, GEMM_DENSE>(p, g, t);
      const int64_t grow = ti.m0 + quarter * 32 + lane;
      // This warp's columns lie in one 128-wide weight block; past N there is
      // none (the partial sums there are zeros), so its multiplier is 1.
      const int64_t nb = (ti.n0 + col_off) >> 7;
      const bool nb_in = nb < nbw;
      float acc[kCols];
#pragma unroll
      for (int i = 0; i < kCols; ++i) acc[i] = 0.0f;
      bool ok = true;
      // The blocks' two multipliers, fetched one block ahead so their latency
      // hides behind the previous block's promotion; rows past the end hold
      // zeros, give them 1.
      float a_s = (ti.nkb > 0 && grow < p.M) ? sa[grow] : 1.0f;
      float b_s = (ti.nkb > 0 && nb_in) ? sb[nb * kbs] : 1.0f;
      for (int kb = 0; kb < ti.nkb; ++kb, ++gk) {
        const int buf = static_cast<int>(gk % P);
        float a_next = 1.0f, b_next = 1.0f;
        if (kb + 1 < ti.nkb) {
          a_next = grow < p.M ? sa[(kb + 1) * p.M + grow] : 1.0f;
          b_next = nb_in ? sb[nb * kbs + kb + 1] : 1.0f;
        }
        if (!wait_or_abort(&part_full[buf], static_cast<uint32_t>((gk / P) & 1), p, s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const float f = 1.0f / (a_s * b_s);
        const uint32_t taddr =
            tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(buf * BN + col_off);
        // One chunk of columns per TMEM load, within the register budget:
        // at BN = 256 eighteen warps leave 96 registers a thread for 64 FP32
        // sums and an 8-column chunk (ten warps holding 128 sums each, or
        // 16-column chunks here, spilled and ran 4-8% slower); at BN = 128
        // ten warps hold 64 sums and 32-column chunks.
        constexpr int kChunk = BN == 256 ? 8 : 32;
#pragma unroll
        for (int ch = 0; ch < kCols / kChunk; ++ch) {
          uint32_t pr[kChunk];
          if constexpr (kChunk == 32) tmem_ld_32x32b_x32(taddr + ch * kChunk, pr);
          else if constexpr (kChunk == 16) tmem_ld_32x32b_x16(taddr + ch * kChunk, pr);
          else tmem_ld_32x32b_x8(taddr + ch * kChunk, pr);
          tmem_ld_wait();
          // Packed FP32 FMAs (two round-to-nearest FMAs per instruction).
#pragma unroll
          for (int i = 0; i < kChunk; i += 2) {
            const float2 s2 = __ffma2_rn(make_float2(__uint_as_float(pr[i]), __uint_as_float(pr[i + 1])),
                                         make_float2(f, f), make_float2(acc[ch * kChunk + i], acc[ch * kChunk + i + 1]));
            acc[ch * kChunk + i] = s2.x;
            acc[ch * kChunk + i + 1] = s2.y;
          }
        }
        tc_fence_before_sync();
        mbar_arrive(&part_empty[buf]);
        a_s = a_next;
        b_s = b_next;
      }
      if (!ok) break;
      store_tile<GEMM_DENSE, kCols>(p, ti, reinterpret_cast<const uint32_t*>(acc), quarter, lane, kCols / 32,
                                    col_off, stg, &tmap_c);
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  pdl_launch_dependents();  // this CTA's tiles are done
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

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

mx_status encode(CUtensorMap* map, CUtensorMapDataType dt, cuuint32_t rank, const void* base, const cuuint64_t* dims,
                 const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swz,
                 CUtensorMapL2promotion l2, const char* what) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return MX_ERR_CUDA;
  }
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, dt, rank, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swz, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled (%s) failed (%d)", what, static_cast<int>(r));
    return MX_ERR_CUDA;
  }
  return MX_OK;
}

// 2-D map over an E4M3 matrix [rows, k] (pitch ld bytes), box 128 K x box_rows,
// 128-byte swizzle, zero fill outside.
mx_status make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t k, int64_t ld, int box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "operand");
}

// 2-D map over a swizzled scale buffer viewed as [atoms][128 x 32-bit words];
// one box is one 512-byte atom.
mx_status make_scale_map(CUtensorMap* map, const void* base, int64_t rows, int64_t k) {
  const int64_t atoms = (rows + 127) / 128 * ((k + 127) / 128);
  cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(atoms)};
  cuuint64_t strides[1] = {512};
  cuuint32_t box[2] = {128, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "scales");
}

// 3-D map over the BF16 output viewed as [groups, rows, N] (row pitch ldc
// elements, group pitch rows*ldc), box 32 x 32 x 1, 64-byte swizzle: the
// epilogue's TMA stores clip at N and at each group's last row.
mx_status make_out_map(CUtensorMap* map, void* c, int64_t groups, int64_t rows, int64_t N, int64_t ldc) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(groups)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ldc * 2), static_cast<cuuint64_t>(rows * ldc * 2)};
  cuuint32_t box[3] = {32, 32, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, c, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B,
                CU_TENSOR_MAP_L2_PROMOTION_NONE, "output");
}

void output_map(const GemmLaunch& L, GParams& p, CUtensorMap* mc, int kind) {
  std::memset(mc, 0, sizeof(*mc));
  p.c_tma = 0;
  const int64_t n_out = L.swiglu ? L.N / 2 : L.N;
  // TMA stores clip a row at 16-byte granularity: with a row width that is not
  // a multiple of 8 elements they would also write the first elements of the
  // pitch gap, so such outputs take the plain bounded stores.
  if (p.c_vec && n_out % 8 == 0) {
    const int64_t groups = (kind == GEMM_GROUPED_K) ? L.n_groups : 1;
    if (make_out_map(mc, L.c, groups, L.M, n_out, L.ldc) == MX_OK) p.c_tma = 1;
  }
}

template <int BN, int KIND>
mx_status launch_cfg(const GemmLaunch& L, const GParams& p_in, int64_t tiles_upper, cudaStream_t s) {
  GParams p = p_in;
  CUtensorMap ma, mb, mc;
  mx_status st = make_map(&ma, L.a_data, L.M, L.K, L.a_ld, kBM);
  if (st != MX_OK) return st;
  st = make_map(&mb, L.b_data, L.b_rows_total, L.K, L.b_ld, BN);
  if (st != MX_OK) return st;
  output_map(L, p, &mc, KIND);
  const size_t smem = Cfg<BN>::smem_bytes(KIND != GEMM_DENSE);
  auto kern = mx_gemm_kernel<BN, KIND>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_status(e, "cudaFuncSetAttribute(smem)");
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(tiles_upper, sm_count()));
  return cuda_status(launch_kernel(kern, static_cast<unsigned>(grid), kThreads, smem, s, 1, ma, mb, mc, p),
                     "mx_gemm launch");
}

// Upper bound of the 256 x bn pair tiles (rows-ragged: one partial tile per
// expert at most).
int64_t pair_tiles_upper(const GemmLaunch& L, int bn = 256) {
  const int64_t nt = (L.N + bn - 1) / bn;
  const int64_t mu = ((L.M + kBM - 1) / kBM + 1) / 2;
  if (L.kind == GEMM_GROUPED_M) return (mu + L.n_groups) * nt;
  if (L.kind == GEMM_GROUPED_K) return mu * nt * L.n_groups;
  return mu * nt;
}

// Dense pair schedule: whole 256 x 256 tiles round by round and, when the last
// round is partial, optionally the split tail (see GParams). Times are
// estimates from the per-SM-pair MXFP8 rate (19 TFLOP/s per SM) and a fixed
// ~1 us per tile (accumulator drain, epilogue). The split costs ~16 us on top
// of its runs (up to two segments per run, each starting its pipeline cold and
// storing a 256 KB FP32 partial; the reduction launch) plus ~0.06 us per
// partial read back, as measured on GB300; runs are at least four K blocks
// long. It therefore pays for few-tile, long-K GEMMs (weight gradients over
// many tokens), not for a short tail of a many-round GEMM.
struct PairPlan {
  int64_t clusters = 1;
  int64_t sk_first = 0, sk_total = 0, tail_tiles = 0;
  int32_t sk_w = 0, sk_slots = 0;
  double est_us = 0.0;
  size_t ws_bytes = 0;
};

int env_int(const char* name, int dflt);

PairPlan plan_pair_dense(const GemmLaunch& L, bool allow_split) {
  static const int split_mode = env_int("MXFP8_GEMM_SPLIT", 1);  // 0: whole tiles only
  if (split_mode == 0) allow_split = false;
  PairPlan pl;
  const int64_t slots = std::max(1, sm_count() / 2);
  const int64_t nt = (L.N + PairCfg::BN - 1) / PairCfg::BN;
  const int64_t tiles = ((L.M + kBM - 1) / kBM + 1) / 2 * nt;
  const int64_t nkb = (L.K + kBK - 1) / kBK;
  const double t_kb = 2.0 * PairCfg::BN * PairCfg::BN * kBK / (2 * 19.0e12) * 1e6;
  const double c_tile = 1.0;
  const int64_t full = tiles / slots, rem = tiles % slots;
  pl.clusters = std::max<int64_t>(1, std::min(tiles, slots));
  pl.est_us = static_cast<double>(full + (rem ? 1 : 0)) * (nkb * t_kb + c_tile);
  if (!allow_split || rem == 0 || nkb < 2) return pl;
  const int64_t total = rem * nkb;
  // <= nkb (rem < slots; a run spans at most two tiles)
  const int64_t w = std::min(nkb, std::max<int64_t>(4, (total + slots - 1) / slots));
  const int64_t runs = (total + w - 1) / w;
  const double split_tail = w * t_kb + 16.0 + 0.06 * static_cast<double>(runs + rem);
  const double whole_tail = nkb * t_kb + c_tile;
  if (split_tail + 4.0 >= whole_tail) return pl;
  pl.clusters = slots;  // runs past `runs` are empty
  pl.sk_first = full * slots;
  pl.sk_total = total;
  pl.tail_tiles = rem;
  pl.sk_w = static_cast<int32_t>(w);
  pl.sk_slots = static_cast<int32_t>(slots);
  pl.est_us = static_cast<double>(full) * (nkb * t_kb + c_tile) + split_tail;
  pl.ws_bytes = static_cast<size_t>(2 * slots) * kPartialFloats * sizeof(float);
  return pl;
}

// The split tail runs only in a workspace the caller passed (large enough).
bool split_allowed(const GemmLaunch& L, size_t need) { return L.ws && L.ws_bytes >= need; }

// The launch arguments live in a per-thread buffer (about 4 KB) rather than
// on the host stack; cudaLaunchKernelEx copies them at the call.
PairArgs* pair_args_scratch() {
  static thread_local PairArgs args;
  return &args;
}

template <int KIND, int kSwiGLU = 0, int BN = 256, bool kTS = false>
mx_status launch_pair(const GemmLaunch& L, const GParams& p_in, cudaStream_t s) {
  GParams p = p_in;
  CUtensorMap ma, mb, msa, msb, mc;
  std::memset(&msa, 0, sizeof(msa));
  std::memset(&msb, 0, sizeof(msb));
  mx_status st = make_map(&ma, L.a_data, L.M, L.K, L.a_ld, kBM);
  if (st != MX_OK) return st;
  st = make_map(&mb, L.b_data, L.b_rows_total, L.K, L.b_ld, BN / 2);
  if (st != MX_OK) return st;
  if constexpr (kTS) {
    // one FP32 scale per tensor (per expert for the stacked weights)
    p.ts_a = static_cast<const float*>(L.a_scale);
    p.ts_b = static_cast<const float*>(L.b_scale);
  } else {
    st = make_scale_map(&msa, L.a_scale, L.M, L.K);
    if (st != MX_OK) return st;
    // Stacked experts: one [E x row atoms x K atoms] view of all experts' scales.
    const int64_t sfb_rows = (KIND == GEMM_GROUPED_M) ? L.n_groups * ((L.N + 127) / 128 * 128) : L.N;
    st = make_scale_map(&msb, L.b_scale, sfb_rows, L.K);
    if (st != MX_OK) return st;
  }
  output_map(L, p, &mc, KIND);
  const size_t smem = PairCfgT<BN, kTS, KIND != GEMM_DENSE>::smem_bytes();
  auto kern = mx_gemm_pair_kernel<KIND, kSwiGLU, false, BN, kTS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_status(e, "cudaFuncSetAttribute(pair smem)");
  int64_t clusters = std::max<int64_t>(1, std::min<int64_t>(pair_tiles_upper(L, BN), sm_count() / 2));
  PairPlan pl;
  if constexpr (KIND == GEMM_DENSE && BN == 256 && !kTS) {
    pl = plan_pair_dense(L, true);
    if (pl.sk_w > 0 && !split_allowed(L, pl.ws_bytes)) pl = plan_pair_dense(L, false);
    if (pl.sk_w > 0) {
      p.ws = static_cast<float*>(L.ws);
      p.sk_first = pl.sk_first;
      p.sk_total = pl.sk_total;
      p.sk_w = pl.sk_w;
      p.sk_slots = pl.sk_slots;
    }
    clusters = pl.clusters;
  }
  PairArgs* args = pair_args_scratch();
  std::memset(args, 0, sizeof(PairArgs));
  args->prob[0] = PairProblem{ma, mb, msa, msb, mc, p};
  args->q = QOut{static_cast<uint8_t*>(L.q_row_data), static_cast<uint8_t*>(L.q_row_scale),
                 static_cast<uint8_t*>(L.q_col_data), static_cast<uint8_t*>(L.q_col_scale)};
  args->n = 1;
  st = cuda_status(launch_kernel(kern, static_cast<unsigned>(2 * clusters), kPairThreads, smem, s, 2, *args),
                   "mx_gemm launch (CTA pairs)");
  if (st == MX_OK && p.sk_w > 0)
    st = cuda_status(launch_kernel(mx_gemm_sk_reduce_kernel, static_cast<unsigned>(32 * pl.tail_tiles), 256, 0, s, 1, p),
                     "mx_gemm split-tail reduction launch");
  return st;
}

// Dispatch overrides (MXFP8_GEMM_PAIR, _BN, _SPLIT, _SCHEDULE) for measuring
// one configuration against another. They exist only in a library built with
// MXFP8_DISPATCH_OVERRIDES defined; the default build ignores the environment
// here, so a stray variable cannot change which kernel runs.
int env_int(const char* name, int dflt) {
#ifdef MXFP8_DISPATCH_OVERRIDES
  const char* v = std::getenv(name);
  return (v && *v) ? std::atoi(v) : dflt;
#else
  (void)name;
  return dflt;
#endif
}

// Dense tile configurations and their estimated time: rounds of tiles over
// the SMs (or pairs of SMs) times the tile's FLOPs at that configuration's
// per-SM rate, plus a fixed per-round cost (accumulator drain, epilogue).
// Rates measured on GB300 with long contractions: CTA pairs 19, single-CTA
// 128 x 256 tiles 16, 128 x 128 tiles 11.2 TFLOP/s per SM.
enum DenseCfg { CFG_PAIR = 0, CFG_BN256 = 1, CFG_BN128 = 2 };

double dense_cfg_time_us(const GemmLaunch& L, int cfg) {
  const int sms = sm_count();
  const int64_t kpad = (L.K + kBK - 1) / kBK * kBK;
  const int64_t mt = (L.M + kBM - 1) / kBM;
  int64_t tiles, slots;
  double tile_flops, rate;
  if (cfg == CFG_PAIR) {
    const PairPlan pl = plan_pair_dense(L, true);
    return (pl.sk_w > 0 && split_allowed(L, pl.ws_bytes)) ? pl.est_us : plan_pair_dense(L, false).est_us;
  } else {
    const int bn = cfg == CFG_BN256 ? 256 : 128;
    tiles = mt * ((L.N + bn - 1) / bn);
    slots = sms;
    tile_flops = 2.0 * kBM * bn * kpad;
    rate = cfg == CFG_BN256 ? 16.0e12 : 11.2e12;
  }
  const int64_t rounds = (tiles + slots - 1) / std::max<int64_t>(slots, 1);
  return static_cast<double>(rounds) * (tile_flops / rate * 1e6 + 1.0);
}

int choose_dense_cfg(const GemmLaunch& L) {
  // MXFP8_GEMM_PAIR (measurement builds): 0 no pairs, 2 force pairs.
  static const int pair_mode = env_int("MXFP8_GEMM_PAIR", 1);
  static const int forced_bn = env_int("MXFP8_GEMM_BN", 0);
  if (pair_mode == 2 && L.N > 128) return CFG_PAIR;
  if (forced_bn == 256) return CFG_BN256;
  if (forced_bn == 128) return CFG_BN128;
  int best = CFG_BN128;
  double best_t = dense_cfg_time_us(L, CFG_BN128);
  for (int cfg : {CFG_BN256, CFG_PAIR}) {
    if (cfg == CFG_PAIR && (pair_mode == 0 || L.N <= 128)) continue;
    if (cfg == CFG_BN256 && L.N <= 128) continue;
    const double t = dense_cfg_time_us(L, cfg);
    if (t < best_t) {
      best_t = t;
      best = cfg;
    }
  }
  return best;
}

// Grouped kinds: 256-wide tiles unless N fits one 128-wide tile.
int choose_bn(const GemmLaunch& L) {
  static const int forced = env_int("MXFP8_GEMM_BN", 0);
  if (forced == 128 || forced == 256) return forced;
  return L.N <= 128 ? 128 : 256;
}

// Grouped kinds on CTA pairs when their 256 x 256 tiles still give every SM work.
bool use_pairs(const GemmLaunch& L) {
  static const int mode = env_int("MXFP8_GEMM_PAIR", 1);
  if (mode == 0 || L.N <= 128) return false;
  if (mode >= 2) return true;
  return pair_tiles_upper(L) >= sm_count() / 2;
}

template <int BN>
mx_status launch_blockwise_bn(const GemmLaunch& L, GParams p, cudaStream_t s) {
  using C = BwCfg<BN>;
  CUtensorMap ma, mb, mc;
  mx_status st = make_map(&ma, L.a_data, L.M, L.K, L.a_ld, kBM);
  if (st != MX_OK) return st;
  st = make_map(&mb, L.b_data, L.N, L.K, L.b_ld, BN);
  if (st != MX_OK) return st;
  output_map(L, p, &mc, GEMM_DENSE);
  const size_t smem = C::smem_bytes();
  auto kern = mx_gemm_blockwise_kernel<BN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_status(e, "cudaFuncSetAttribute(blockwise smem)");
  const int64_t tiles = (L.M + kBM - 1) / kBM * ((L.N + BN - 1) / BN);
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(tiles, sm_count()));
  return cuda_status(launch_kernel(kern, static_cast<unsigned>(grid), C::kThreads, smem, s, 1, ma, mb, mc, p,
                                   L.bw_a_scale, L.bw_b_scale),
                     "mx_gemm_fp8_blockwise launch");
}

// 128 x 256 tiles unless N fits one 128-wide tile.
mx_status launch_blockwise(const GemmLaunch& L, GParams p, cudaStream_t s) {
  return L.N > 128 ? launch_blockwise_bn<256>(L, p, s) : launch_blockwise_bn<128>(L, p, s);
}

}  // namespace

// Scratch memory of mx_gemm_static_workspace: a fixed array in device memory,
// reserved when the library's kernels are loaded on a device and held until
// the process exits, for callers that may not allocate. Every call uses the
// same array.
static __device__ __align__(256) float g_static_ws[MX_STATIC_WORKSPACE_BYTES / sizeof(float)];

mx_status static_workspace(void** ptr, size_t* bytes) {
  // Host code cannot use g_static_ws's name as a device address: the address
  // comes from the runtime, once per device, with that device current.
  static std::mutex mu;
  static void* cache[64] = {nullptr};
  int dev = 0;
  mx_status st = cuda_status(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != MX_OK) return st;
  if (dev < 0 || dev >= 64) {
    set_error("device ordinal %d is outside the static workspace table", dev);
    return MX_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    st = cuda_status(cudaGetSymbolAddress(&p, g_static_ws), "cudaGetSymbolAddress(static workspace)");
    if (st != MX_OK) return st;
    cache[dev] = p;
  }
  *ptr = cache[dev];
  *bytes = MX_STATIC_WORKSPACE_BYTES;
  return MX_OK;
}

size_t gemm_workspace_bytes(const GemmLaunch& L) {
  if (L.kind != GEMM_DENSE || L.swiglu || L.bw_a_scale || L.tensor_scaled || L.M == 0 || L.N == 0 || L.K == 0)
    return 0;
  GemmLaunch q = L;
  q.ws = reinterpret_cast<void*>(uintptr_t{16});  // any workspace: the size a split would need
  q.ws_bytes = SIZE_MAX;
  if (choose_dense_cfg(q) != CFG_PAIR) return 0;
  const PairPlan pl = plan_pair_dense(q, true);
  return pl.sk_w > 0 ? pl.ws_bytes : 0;
}

namespace {

GParams make_gparams(const GemmLaunch& L) {
  GParams p;
  p.a_scale = static_cast<const uint8_t*>(L.a_scale);
  p.b_scale = static_cast<const uint8_t*>(L.b_scale);
  p.M = L.M;
  p.N = L.N;
  p.n_out = L.swiglu ? L.N / 2 : L.N;
  p.K = L.K;
  p.ka = (L.K + 127) / 128;
  p.a_ra = (L.M + 127) / 128;
  p.b_rows_group = L.N;
  p.b_ra = (L.N + 127) / 128;
  p.b_scale_stride = static_cast<int64_t>(mx_scale_bytes(L.N, L.K));
  p.c = static_cast<__nv_bfloat16*>(L.c);
  p.ldc = L.ldc;
  p.c_group_stride = L.M * L.ldc;
  p.c_vec = ((reinterpret_cast<uintptr_t>(L.c) & 15u) == 0 && L.ldc % 8 == 0) ? 1 : 0;
  p.c_tma = 0;
  // Walk N first when A is the larger operand (and always for the rows-ragged
  // grouped GEMM): the CTAs that share an A tile then run at the same time and
  // A leaves HBM once, while the smaller B stays resident in L2.
  p.n_fast = (L.kind == GEMM_GROUPED_M || (L.kind == GEMM_DENSE && L.M >= L.N)) ? 1 : 0;
  p.offsets = L.offsets;
  p.n_groups = L.n_groups;
  p.dev_status = L.dev_status;
  p.timeout_ns = wait_timeout_ns();
  p.sk_first = 0;
  p.sk_total = 0;
  p.sk_w = 0;
  p.sk_slots = 0;
  p.ws = nullptr;
  p.ts_a = nullptr;
  p.ts_b = nullptr;
  p.q_cap = L.q_row_data ? L.q_cap : 0;
  return p;
}

// Cost of one pair tile of L in 128-K blocks, plus the per-tile drain and
// epilogue (about two blocks' time).
int64_t pair_tile_cost(const GemmLaunch& L) { return (L.K + kBK - 1) / kBK + 2; }

// Greedy longest-first schedule of the problems' tiles over `clusters` SM
// pairs (problems already in decreasing tile cost): every tile goes to the
// cluster that would finish first. Fills args->cnt; returns the latest
// finish, or -1 if a count does not fit the table.
int64_t schedule_greedy(PairArgs* args, const GemmLaunch* Ls, int n, int64_t clusters) {
  std::vector<int64_t> load(static_cast<size_t>(clusters), 0);
  using Slot = std::pair<int64_t, int64_t>;  // (load, cluster): ties go to the lower index
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
  for (int64_t c = 0; c < clusters; ++c) heap.push({0, c});
  for (int i = 0; i < n; ++i) {
    const int64_t cost = pair_tile_cost(Ls[i]);
    std::vector<int64_t> cnt(static_cast<size_t>(clusters), 0);
    for (int64_t t = 0; t < pair_tiles_upper(Ls[i]); ++t) {
      Slot sl = heap.top();
      heap.pop();
      ++cnt[static_cast<size_t>(sl.second)];
      sl.first += cost;
      heap.push(sl);
    }
    for (int64_t c = 0; c < clusters; ++c) {
      if (cnt[static_cast<size_t>(c)] > 255) return -1;
      args->cnt[i][c] = static_cast<uint8_t>(cnt[static_cast<size_t>(c)]);
    }
  }
  int64_t worst = 0;
  while (!heap.empty()) {
    worst = std::max(worst, heap.top().first);
    heap.pop();
  }
  return worst;
}

// Latest finish of round-robin: cluster c takes launch tiles c, c + clusters, ...
int64_t schedule_round_robin(const GemmLaunch* Ls, int n, int64_t clusters) {
  std::vector<int64_t> load(static_cast<size_t>(clusters), 0);
  int64_t t = 0;
  for (int i = 0; i < n; ++i) {
    const int64_t cost = pair_tile_cost(Ls[i]);
    for (int64_t j = 0; j < pair_tiles_upper(Ls[i]); ++j, ++t) load[static_cast<size_t>(t % clusters)] += cost;
  }
  return *std::max_element(load.begin(), load.end());
}

// Several dense GEMMs in one launch of the pair kernel.
mx_status launch_pair_multi(const GemmLaunch* Ls_in, int n, cudaStream_t s) {
  constexpr int BN = 256;
  // Block-scaled problems, or (all of them) one FP32 scale per tensor.
  const bool ts = Ls_in[0].tensor_scaled;
  for (int i = 1; i < n; ++i)
    if (Ls_in[i].tensor_scaled != ts) {
      set_error("several GEMMs per launch: block-scaled and tensor-scaled problems do not mix");
      return MX_ERR_INVALID_ARG;
    }
  PairArgs* args = pair_args_scratch();
  std::memset(args, 0, sizeof(PairArgs));
  // Longest tiles first: they start early and the short ones fill in behind.
  GemmLaunch Ls[kMaxProblems];
  for (int i = 0; i < n; ++i) Ls[i] = Ls_in[i];
  std::stable_sort(Ls, Ls + n, [](const GemmLaunch& a, const GemmLaunch& b) {
    return pair_tile_cost(a) > pair_tile_cost(b);
  });
  int64_t tiles = 0;
  for (int i = 0; i < n; ++i) {
    const GemmLaunch& L = Ls[i];
    PairProblem& pr = args->prob[i];
    pr.p = make_gparams(L);
    mx_status st = make_map(&pr.a, L.a_data, L.M, L.K, L.a_ld, kBM);
    if (st != MX_OK) return st;
    st = make_map(&pr.b, L.b_data, L.b_rows_total, L.K, L.b_ld, BN / 2);
    if (st != MX_OK) return st;
    if (ts) {
      pr.p.ts_a = static_cast<const float*>(L.a_scale);
      pr.p.ts_b = static_cast<const float*>(L.b_scale);
    } else {
      st = make_scale_map(&pr.sfa, L.a_scale, L.M, L.K);
      if (st != MX_OK) return st;
      st = make_scale_map(&pr.sfb, L.b_scale, L.N, L.K);
      if (st != MX_OK) return st;
    }
    output_map(L, pr.p, &pr.c, GEMM_DENSE);
    args->tile0[i] = tiles;
    tiles += pair_tiles_upper(L);
  }
  args->tile0[n] = tiles;
  args->n = n;
  const size_t smem = ts ? PairCfgT<BN, true, false>::smem_bytes() : PairCfgT<BN, false, false>::smem_bytes();
  auto kern = ts ? mx_gemm_pair_kernel<GEMM_DENSE, 0, true, BN, true>
                 : mx_gemm_pair_kernel<GEMM_DENSE, 0, true, BN, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_status(e, "cudaFuncSetAttribute(pair smem)");
  const int64_t clusters = std::max<int64_t>(1, std::min<int64_t>(tiles, sm_count() / 2));
  // The balanced schedule where it finishes clearly earlier than round-robin
  // (same tiles, same results; only the order of work changes).
  static const int sched_mode = env_int("MXFP8_GEMM_SCHEDULE", 1);  // 0: round-robin only
  if (sched_mode != 0 && clusters <= kMaxSchedClusters) {
    const int64_t greedy = schedule_greedy(args, Ls, n, clusters);
    const int64_t rr = schedule_round_robin(Ls, n, clusters);
    args->sched = (greedy > 0 && greedy * 100 < rr * 97) ? 1 : 0;
  }
  return cuda_status(launch_kernel(kern, static_cast<unsigned>(2 * clusters), kPairThreads, smem, s, 2, *args),
                     "mx_gemm_multi launch (CTA pairs)");
}


}  // namespace

mx_status launch_gemm(const GemmLaunch& L, cudaStream_t s) {
  if (L.M == 0 || L.N == 0) return MX_OK;
  if (L.kind != GEMM_DENSE && L.n_groups > kMaxGroups) {
    set_error("mx_grouped_gemm: at most %d groups", kMaxGroups);
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  if (L.kind == GEMM_GROUPED_K && L.n_groups == 0) return MX_OK;
  GParams p = make_gparams(L);

  if (L.bw_a_scale) return launch_blockwise(L, p, s);
  if (L.tensor_scaled) {
    // one FP32 scale per tensor / per expert: 256 x 256 pair tiles, two accumulators
    if (L.kind == GEMM_DENSE) return launch_pair<GEMM_DENSE, 0, 256, true>(L, p, s);
    if (L.kind == GEMM_GROUPED_M) return launch_pair<GEMM_GROUPED_M, 0, 256, true>(L, p, s);
    return launch_pair<GEMM_GROUPED_K, 0, 256, true>(L, p, s);
  }
  if (L.swiglu) return L.q_row_data ? launch_pair<GEMM_GROUPED_M, 2>(L, p, s) : launch_pair<GEMM_GROUPED_M, 1>(L, p, s);
  int bn;
  if (L.kind == GEMM_DENSE) {
    const int cfg = choose_dense_cfg(L);
    if (cfg == CFG_PAIR) return launch_pair<GEMM_DENSE>(L, p, s);
    bn = cfg == CFG_BN256 ? 256 : 128;
  } else {
    if (use_pairs(L))
      return L.kind == GEMM_GROUPED_K ? launch_pair<GEMM_GROUPED_K>(L, p, s) : launch_pair<GEMM_GROUPED_M>(L, p, s);
    bn = choose_bn(L);
  }
  const int64_t mt = (L.M + kBM - 1) / kBM;
  const int64_t nt = (L.N + bn - 1) / bn;
  int64_t tiles_upper = mt * nt;
  if (L.kind == GEMM_GROUPED_M) tiles_upper = (mt + L.n_groups) * nt;
  if (L.kind == GEMM_GROUPED_K) tiles_upper = static_cast<int64_t>(L.n_groups) * mt * nt;

  switch (L.kind) {
    case GEMM_DENSE:
      return bn == 256 ? launch_cfg<256, GEMM_DENSE>(L, p, tiles_upper, s)
                       : launch_cfg<128, GEMM_DENSE>(L, p, tiles_upper, s);
    case GEMM_GROUPED_M:
      return bn == 256 ? launch_cfg<256, GEMM_GROUPED_M>(L, p, tiles_upper, s)
                       : launch_cfg<128, GEMM_GROUPED_M>(L, p, tiles_upper, s);
    default:
      return bn == 256 ? launch_cfg<256, GEMM_GROUPED_K>(L, p, tiles_upper, s)
                       : launch_cfg<128, GEMM_GROUPED_K>(L, p, tiles_upper, s);
  }
}

mx_status launch_gemm_multi(const GemmLaunch* Ls, int n, cudaStream_t s) {
  // Problems with nothing to compute drop out; K = 0 is the caller's memset.
  GemmLaunch live[kMaxProblems];
  int m = 0;
  int64_t tiles = 0;
  bool pairs = true;
  for (int i = 0; i < n; ++i) {
    if (Ls[i].M == 0 || Ls[i].N == 0) continue;
    live[m] = Ls[i];
    tiles += pair_tiles_upper(Ls[i]);
    if (Ls[i].kind != GEMM_DENSE || Ls[i].N <= 128) pairs = false;
    ++m;
  }
  if (m == 0) return MX_OK;
  // One pair launch when the problems together fill the SM pairs at least
  // once; otherwise each GEMM on its own best configuration.
  if (m > 1 && pairs && tiles >= sm_count() / 2) return launch_pair_multi(live, m, s);
  for (int i = 0; i < m; ++i) {
    mx_status st = launch_gemm(live[i], s);
    if (st != MX_OK) return st;
  }
  return MX_OK;
}

}  // namespace mx
