// mx_internal.h - declarations shared by the translation units of the library
// (host side only; no device code here).
#pragma once

#include <cuda_runtime.h>
#include <cstdint>
#include <cstring>
#include <utility>

#include "../../include/mxfp8.h"

namespace mx {

// Last error message of this host thread (returned by mx_last_error()).
void set_error(const char* fmt, ...);

// MX_OK if e == cudaSuccess, else records the message and returns MX_ERR_CUDA.
mx_status cuda_status(cudaError_t e, const char* what);

// Bounded-wait limit (nanoseconds) for device-side mbarrier waits. Read once
// from the MXFP8_WAIT_TIMEOUT_NS environment variable (default 2 s).
uint64_t wait_timeout_ns();

// Number of SMs of the current device (cached per device).
int sm_count();

// Programmatic dependent launch on (default); MXFP8_PDL=0 turns it off.
bool pdl_enabled();

// Launches kern on stream s. With programmatic stream serialization the grid
// may be scheduled while the kernel before it on the stream is finishing; each
// kernel of this library runs griddepcontrol.wait before its first global
// memory access, which returns once that previous grid has completed and its
// writes are visible, and griddepcontrol.launch_dependents at its start.
// cluster_x > 1 also sets the cluster shape.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t s,
                          unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  std::memset(attr, 0, sizeof(attr));
  unsigned n = 0;
  if (pdl_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// --- quantiser -------------------------------------------------------------
struct QuantLaunch {
  const void* x;
  int64_t rows, cols, ldx;
  void* row_data;
  void* row_scale;
  void* col_data;
  void* col_scale;
  const int64_t* offsets;  // nullptr: dense column copy
  int n_groups;
  int64_t col_pitch;       // rows (dense) or the grouped capacity
  int64_t batch;           // stacked matrices (1 unless batched)
  int64_t x_batch_stride;  // elements between stacked inputs
  bool x_f32 = false;      // FP32 input (else BF16)
  int* dev_status;
};
mx_status launch_quantize(const QuantLaunch& q, bool do_row, bool do_col, cudaStream_t s);
// Several dense BF16 matrices (batch 1 each, no groups) in one launch.
mx_status launch_quantize_multi(const QuantLaunch* qs, int n, bool do_row, bool do_col, cudaStream_t s);
// Current scaling: amax of each matrix of the stack q (zeroed first, then
// reduced), and the quantisation with scale[b] = amax[b] / format_max (1 for an
// invalid amax), written to `scale`.
mx_status launch_current_amax(const QuantLaunch& q, float* amax, cudaStream_t s);
mx_status launch_quantize_current(const QuantLaunch& q, const float* amax, float format_max, float* scale,
                                  bool do_row, bool do_col, cudaStream_t s);
// Blockwise FP8 variant: block = 1 (1 x 128 activation blocks, scale[kb][rows])
// or 128 (128 x 128 weight blocks, scale[row block][kb]).
mx_status launch_quantize_blockwise(const void* x, int64_t rows, int64_t cols, int64_t ldx, int block, void* data,
                                    float* scale, cudaStream_t s);

// --- GEMM ------------------------------------------------------------------
enum GemmKind { GEMM_DENSE = 0, GEMM_GROUPED_M = 1, GEMM_GROUPED_K = 2 };

struct GemmLaunch {
  GemmKind kind;
  const void* a_data;
  const void* a_scale;
  int64_t a_ld;
  const void* b_data;
  const void* b_scale;
  int64_t b_ld;
  int64_t M;        // rows of C (per group for GROUPED_K)
  int64_t N;        // columns of C
  int64_t K;        // contraction length (capacity for GROUPED_K)
  int64_t b_rows_total;  // rows of the 2-D view of b (E*N for GROUPED_M, else N)
  void* c;
  int64_t ldc;
  const int64_t* offsets;
  int n_groups;
  int* dev_status;
  bool swiglu = false;  // rows-ragged only: C = SwiGLU(A . B^T), gate = B rows [0, N/2), up = [N/2, N)
  // Blockwise FP8 variant (dense): FP32 multipliers of A's 1 x 128 blocks
  // ([K/128][M]) and B's 128 x 128 blocks ([ceil(N/128)][K/128]); a_scale /
  // b_scale unused.
  const float* bw_a_scale = nullptr;
  const float* bw_b_scale = nullptr;
  // The caller's workspace for the dense split tail; without one (or with
  // too small a one) the GEMM runs whole tiles only.
  void* ws = nullptr;
  size_t ws_bytes = 0;
  // Current-scaling recipe: a_scale / b_scale are FP32 tensor scales (b: one
  // per expert for rows-ragged grouped GEMMs) applied in the epilogue.
  bool tensor_scaled = false;
  // Rows-ragged SwiGLU only: instead of the BF16 output, its MX copies as
  // mx_quantize (both copies, per-expert column segments) would write them from
  // that output: row copy [M, N/2] + scales, column copy [N/2, q_cap] + scales.
  void* q_row_data = nullptr;
  void* q_row_scale = nullptr;
  void* q_col_data = nullptr;
  void* q_col_scale = nullptr;
  int64_t q_cap = 0;
};
mx_status launch_gemm(const GemmLaunch& g, cudaStream_t s);
// Bytes of workspace the dense GEMM L would use for its split tail (0: none).
size_t gemm_workspace_bytes(const GemmLaunch& L);
// Device address and size of the library's static scratch array on the
// current device (looked up on the first call per device).
mx_status static_workspace(void** ptr, size_t* bytes);
// Up to MX_MAX_GEMM_MULTI independent dense GEMMs; one launch of the pair
// kernel when they fill the GPU together, else one launch each.
mx_status launch_gemm_multi(const GemmLaunch* Ls, int n, cudaStream_t s);

}  // namespace mx
