/*
 * mxfp8.h - C ABI of the MXFP8 block-scaled quantiser, GEMM and grouped GEMM
 * for NVIDIA GB300 (sm_103a).
 *
 * The operations follow two web pages that describe MXFP8 training of linear
 * and MoE-expert layers:
 *   [DSV3] "DeepSeek-V3 16B FSDP2 MXFP8/HiF8 训练设计" (hyper-parallel issue #329)
 *   [TT]   "低精度训练特性（MXFP8 / HiFloat8）" (torchtitan-npu)
 * and one page on number formats:
 *   [FMT]  "浮点格式、数值稳定性与混合精度" (arganzheng.life)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All pointers named *_data, *_scale, x, c, workspace and group_offsets are
 *   DEVICE pointers, allocated and owned by the caller. The library never
 *   allocates or frees device memory. Scratch memory is the caller's buffer
 *   (mx_gemm_with_workspace, sized by mx_gemm_workspace_bytes), except for
 *   mx_gemm_static_workspace, whose scratch is one fixed array of
 *   MX_STATIC_WORKSPACE_BYTES that the library declares in device memory
 *   (held on every device that loads the library's kernels). No other state
 *   is kept between calls.
 * - Work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *   void*; NULL is the legacy default stream) on the current device, which must
 *   be an sm_103 GPU. Nothing is synchronised. Kernels are launched with
 *   programmatic stream serialization: one may be scheduled while the kernel
 *   before it on the stream finishes, but it reads and writes memory only once
 *   that kernel has completed, so stream order is what the caller sees
 *   (environment MXFP8_PDL=0 launches without it).
 * - Every call validates its arguments on the host first; on failure it
 *   returns a non-OK status and launches nothing. There is no fallback to any
 *   other kernel or precision ([DSV3] §13.4 and §15: a failure must be raised,
 *   never replaced by a high-precision GEMM).
 * - Grouped calls (mx_quantize with group offsets, mx_grouped_gemm,
 *   mx_grouped_gemm_swiglu) take at most MX_MAX_GROUPS groups; more is
 *   MX_ERR_UNSUPPORTED_SHAPE on the host, before anything is launched. (The
 *   kernels keep every group's offsets in shared memory beside the operand
 *   pipeline.)
 * - Environment: MXFP8_PDL=0 launches without programmatic dependent launch;
 *   MXFP8_WAIT_TIMEOUT_NS bounds every device-side wait (default 2 s, at
 *   least 1 ms). Nothing else in the environment changes what the library
 *   does. (A library built with MXFP8_DISPATCH_OVERRIDES defined, for
 *   measurements only, also reads MXFP8_GEMM_PAIR, MXFP8_GEMM_BN,
 *   MXFP8_GEMM_SPLIT and MXFP8_GEMM_SCHEDULE to force a GEMM configuration;
 *   the default build ignores them.)
 * - `dev_status` (device int*, may be NULL): checks that only the device can
 *   make (group offsets) and bounded waits that expire write a non-zero
 *   mx_status value there; the kernels never trap. The caller zeroes it
 *   before the call and reads it after synchronising. The host-side return
 *   value cannot report these.
 *
 * Data formats ([DSV3] §3, §3.1; [TT] 线性层低精度; [FMT] §二.2)
 * -------------------------------------------------------------
 * - Input: BF16, row-major.
 * - Data: E4M3 codes (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no
 *   infinities, S.1111.111 is NaN, largest finite 448), one byte per element.
 * - Scales: E8M0 codes (2**(code-127); 0xFF is NaN), one per block of 32
 *   consecutive elements along the contraction dimension.
 * - Scale rule: X = floor(log2(amax)) - 8 clamped to [-127, 127], code = X+127;
 *   element code = E4M3(x * 2**-X) rounded to nearest, ties to even, magnitudes
 *   above 448 saturate. amax = 0 gives code 0x00; a block holding NaN/Inf gives
 *   scale 0xFF and data 0x7F with each element's sign.
 * - Row copy of T[R, C]: 1x32 blocks along each row; data [R, C].
 * - Column copy of T[R, C]: 32x1 blocks down each column, stored TRANSPOSED:
 *   data [C, R], so its blocks are 1x32 along its rows. Every GEMM operand is
 *   therefore K-major with blocks along K.
 *
 * Scale-tile layout (the one the sm_103a block-scaled MMA consumes; the pages
 * describe none): the logical scale matrix S[rows, kb] (kb = ceil(k/32)) is
 * padded with zero bytes to [ceil(rows/128)*128, ceil(kb/4)*4] and cut into
 * 512-byte atoms of 128 rows x 4 scale columns. Atom (ra, ka) = (r/128, k/4)
 * starts at byte (ra * ceil(kb/4) + ka) * 512 (scale-column atoms fastest).
 * Inside an atom the byte of S[r, k] sits at (r%32)*16 + ((r/32)%4)*4 + (k%4),
 * i.e. 32 lines of 16 bytes, line r%32 holding rows r%32, +32, +64, +96.
 * mx_scale_bytes()
 * returns the padded size. Padding bytes are written as 0 by mx_quantize.
 */
#ifndef MXFP8_GB300_H
#define MXFP8_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MXFP8_ABI_VERSION 1

/* Largest n_groups of the grouped calls (see the conventions above). */
#define MX_MAX_GROUPS 512

typedef enum mx_status {
  MX_OK = 0,
  MX_ERR_INVALID_ARG = 1,       /* null pointer, bad enum, negative size, inconsistent operands */
  MX_ERR_UNSUPPORTED_SHAPE = 2, /* a size the kernels do not take (e.g. K not a multiple of 32) */
  MX_ERR_ALIGNMENT = 3,         /* a pointer or pitch is not 16-byte aligned */
  MX_ERR_CUDA = 4,              /* a CUDA call failed; mx_last_error() has the message */
  MX_ERR_DEVICE_CHECK = 5,      /* device-side validation failed (reported via dev_status) */
  MX_ERR_TIMEOUT = 6,           /* a bounded device wait expired (reported via dev_status) */
  MX_ERR_NO_DEVICE = 7          /* the current device is not an sm_103 GPU */
} mx_status;

typedef enum mx_axis {
  MX_ROWWISE = 1, /* 1x32 blocks along rows (the "row" copy of [DSV3] §3.1) */
  MX_COLWISE = 2, /* 32x1 blocks down columns, stored transposed (the "col" copy) */
  MX_BOTH = 3     /* both copies from one read of the input ([DSV3] §8.1 dual-axis) */
} mx_axis;

/* GEMM modes of the direction table in [DSV3] §8 (layouts NT, NN, TN of §13.4).
 * With column copies stored transposed, each mode computes C = A . B^T:
 *   MX_FPROP  Y[M,N]  = X . W^T      a = X row copy [M,K],   b = W row copy [N,K]
 *   MX_DGRAD  dX[M,K] = dY . W       a = dY row copy [M,N],  b = W col copy [K,N]
 *   MX_WGRAD  dW[N,K] = dY^T . X     a = dY col copy [N,M],  b = X col copy [K,M]
 * The mode only selects which operand orientations are accepted. */
typedef enum mx_mode { MX_FPROP = 0, MX_DGRAD = 1, MX_WGRAD = 2 } mx_mode;

/* One quantised operand ([DSV3] §7.4 QuantizedOperand: data, scale, orientation). */
typedef struct mx_operand {
  const void* data;  /* E4M3 codes: row r starts at data + r*ld bytes; k contiguous */
  const void* scale; /* swizzled E8M0 scales of the logical [rows, ceil(k/32)] */
  int64_t rows;      /* rows of this operand (M for a, N for b) */
  int64_t k;         /* contraction length (for grouped wgrad: the padded capacity) */
  int64_t ld;        /* bytes between rows, 0 means k; multiple of 16 */
  int32_t orient;    /* MX_ROWWISE or MX_COLWISE: which copy of its source tensor */
  int32_t reserved;  /* must be 0 */
} mx_operand;

/* Size in bytes of the swizzled scale buffer of a [rows, k] operand
 * (ceil(rows/128)*128 * ceil(ceil(k/32)/4)*4). Host-only, pure function. */
size_t mx_scale_bytes(int64_t rows, int64_t k);

/* Total padded length of a grouped column copy: sum over groups of
 * ceil(m_e/128)*128 for m_e = host_offsets[e+1] - host_offsets[e].
 * Returns -1 if the offsets are not non-decreasing from 0. Host pointer. */
int64_t mx_grouped_padded_rows(const int64_t* host_offsets, int n_groups);

/*
 * mx_quantize - dynamic MX quantisation of a BF16 matrix ([DSV3] §8.1, §13.3
 * Quantizer.quantize(tensor, orientation, group_list); [TT] npu_dynamic_mx_quant
 * and, with groups, npu_grouped_dynamic_mx_quant).
 *
 *   x        BF16 [rows, cols], row pitch ldx elements (ldx >= cols); 16-byte aligned,
 *            ldx a multiple of 8.
 *   axis     MX_ROWWISE, MX_COLWISE or MX_BOTH.
 *   Row copy (ROWWISE/BOTH): row_data [rows, cols] E4M3 (pitch cols bytes),
 *            row_scale mx_scale_bytes(rows, cols) bytes. Needs cols % 32 == 0.
 *   Column copy (COLWISE/BOTH), dense (group_offsets == NULL):
 *            col_data [cols, rows] E4M3 (pitch rows bytes), col_scale
 *            mx_scale_bytes(cols, rows) bytes. Needs rows % 32 == 0.
 *   Column copy, grouped (group_offsets != NULL): group e is rows
 *            [off[e], off[e+1]) of x (int64 device array of n_groups+1 entries,
 *            off[0] = 0, non-decreasing, off[n_groups] = rows). 32x1 blocks
 *            restart at each group's first row; group e's segment is padded
 *            with zero codes to a multiple of 128 and starts at column
 *            poff[e] = sum_{i<e} ceil(m_i/128)*128 of col_data [cols, col_capacity]
 *            (pitch col_capacity bytes). col_scale holds
 *            mx_scale_bytes(cols, col_capacity) bytes. col_capacity must be a
 *            multiple of 128 and >= the padded total; columns beyond the padded
 *            total are not written. 1 <= n_groups <= MX_MAX_GROUPS. Bad offsets or too small a capacity are
 *            reported as MX_ERR_DEVICE_CHECK through dev_status and nothing is
 *            written. The row copy is unaffected by groups.
 *   All outputs 16-byte aligned. Unused outputs may be NULL.
 */
mx_status mx_quantize(const void* x, int64_t rows, int64_t cols, int64_t ldx, int axis,
                      void* row_data, void* row_scale, void* col_data, void* col_scale,
                      const int64_t* group_offsets, int n_groups, int64_t col_capacity,
                      int* dev_status, void* stream);

/*
 * mx_quantize_batched - the dense mx_quantize applied in one launch to `batch`
 * matrices stacked in memory, e.g. the per-expert weights [E, N, K] of the
 * routed experts ([DSV3] §5.2: stacked 3-D expert parameters; §8.1: weights
 * are quantised into row and col copies once after each optimizer step).
 *
 *   x          BF16; matrix b is [rows, cols] at x + b*x_batch_stride elements,
 *              row pitch ldx. x_batch_stride >= rows*ldx and a multiple of 8.
 *   row_data   [batch][rows][cols] E4M3 (matrix stride rows*cols bytes);
 *   row_scale  matrix stride mx_scale_bytes(rows, cols) bytes.
 *   col_data   [batch][cols][rows] E4M3 (matrix stride cols*rows bytes);
 *   col_scale  matrix stride mx_scale_bytes(cols, rows) bytes.
 *   Per-matrix layouts, requirements and results are exactly those of the
 *   dense mx_quantize (no groups). batch == 0 is a no-op.
 */
mx_status mx_quantize_batched(const void* x, int64_t batch, int64_t rows, int64_t cols, int64_t ldx,
                              int64_t x_batch_stride, int axis, void* row_data, void* row_scale, void* col_data,
                              void* col_scale, int* dev_status, void* stream);

/*
 * mx_quantize_f32 - the weight refresh: row and column copies generated from
 * FP32 master weights after an optimizer step ("DeepSeek-V3 16B FSDP2
 * MXFP8/HiF8 训练设计" §8.1: weights are quantised once from the FP32 master
 * into row/col data and scales; §10: the step data flow refreshes the MXFP8
 * dual-axis data and E8M0 scales from the new master). The blocks are formed
 * from the FP32 values themselves: no rounding to BF16 happens first, so a
 * value that BF16 cannot hold quantises as itself.
 *
 *   x          FP32; matrix b is [rows, cols] at x + b*x_batch_stride elements,
 *              row pitch ldx elements (ldx >= cols, a multiple of 4);
 *              16-byte aligned; x_batch_stride >= rows*ldx and a multiple of 4
 *              when batch > 1. A single matrix is batch = 1.
 *   Outputs, their layouts and strides, requirements (cols % 32 == 0; rows %
 *   32 == 0 for the column copy), alignment and error reporting are exactly
 *   those of mx_quantize_batched. batch == 0 is a no-op.
 */
mx_status mx_quantize_f32(const float* x, int64_t batch, int64_t rows, int64_t cols, int64_t ldx,
                          int64_t x_batch_stride, int axis, void* row_data, void* row_scale, void* col_data,
                          void* col_scale, int* dev_status, void* stream);

/* One BF16 matrix of an mx_quantize_multi call: the arguments of the dense
 * mx_quantize (no groups), gathered in a struct. */
typedef struct mx_quant_tensor {
  const void* x;    /* BF16 [rows, cols], row pitch ldx elements */
  int64_t rows;
  int64_t cols;
  int64_t ldx;
  void* row_data;   /* [rows, cols] E4M3, or NULL when the row copy is not asked for */
  void* row_scale;  /* mx_scale_bytes(rows, cols) bytes */
  void* col_data;   /* [cols, rows] E4M3, or NULL when the column copy is not asked for */
  void* col_scale;  /* mx_scale_bytes(cols, rows) bytes */
} mx_quant_tensor;

/*
 * mx_quantize_multi - the dense mx_quantize of up to MX_MAX_MULTI unrelated
 * BF16 matrices (different shapes and buffers) in one launch, e.g. the
 * activation X and the weight W that one Linear's forward GEMM reads ([DSV3]
 * §8.1: X and W are both quantised into row and column copies before the
 * forward GEMM; §10, the step data flow). One launch shares the persistent
 * grid's ramp and tail between the matrices; each matrix's results are
 * exactly those of mx_quantize on it alone.
 *
 *   tensors  host array of n descriptors (host pointer; read before return).
 *   n        0 .. MX_MAX_MULTI; n == 0 and matrices with rows == 0 or
 *            cols == 0 are no-ops.
 *   axis     one axis for every matrix (MX_ROWWISE, MX_COLWISE or MX_BOTH).
 *   Requirements per matrix are those of the dense mx_quantize: cols % 32 ==
 *   0, rows % 32 == 0 for the column copy, x 16-byte aligned with ldx % 8 ==
 *   0, outputs 16-byte aligned. Any violation fails the whole call before
 *   anything is launched, with the index of the matrix in mx_last_error().
 *   Output buffers must not overlap one another or any input.
 */
#define MX_MAX_MULTI 8
mx_status mx_quantize_multi(const mx_quant_tensor* tensors, int n, int axis, int* dev_status, void* stream);

/*
 * mx_gemm - block-scaled GEMM C[M,N] = A[M,K] . B[N,K]^T with FP32 accumulation
 * and BF16 output rounded to nearest even ([DSV3] §8 and §13.4
 * low_precision_matmul; [TT] npu_quant_matmul; [FMT] §五.1).
 *
 *   mode     MX_FPROP (a, b row copies), MX_DGRAD (a row, b col copy) or
 *            MX_WGRAD (a, b col copies); a mismatch is MX_ERR_INVALID_ARG.
 *   a, b     operands (host pointers to the structs); M = a->rows,
 *            N = b->rows, K = a->k = b->k, K % 32 == 0. K == 0 writes zeros.
 *   c        BF16 [M, N], row pitch ldc elements (ldc >= N), 2-byte aligned.
 *            With c 16-byte aligned and ldc % 8 == 0 the epilogue uses
 *            16-byte stores; otherwise element stores.
 * Deterministic: no split-K and no atomics, so repeated calls give identical bits.
 */
mx_status mx_gemm(int mode, const mx_operand* a, const mx_operand* b, void* c, int64_t ldc,
                  int* dev_status, void* stream);

/*
 * Scratch memory of the dense GEMM. When the 256 x 256 tiles leave the last
 * round over the GPU's SM pairs mostly empty and the contraction is long
 * (weight gradients over many tokens), the contraction of those last tiles can
 * be cut into equal runs of 128-K blocks, one run per SM pair; each run leaves
 * FP32 partial tiles in a workspace, and a second kernel adds a tile's
 * partials in a fixed order and rounds once to BF16 (so results stay
 * bit-identical from call to call, and within the same error bound as the
 * whole-tile path: FP32 accumulation throughout). mx_gemm never splits;
 * mx_gemm_with_workspace splits when the caller's workspace is large enough
 * and the split is estimated to be faster.
 *
 * mx_gemm_workspace_bytes - bytes of workspace mx_gemm_with_workspace would use
 * for these operands on the current device (0: this GEMM does not split).
 *   Same operand checks as mx_gemm; *bytes is a host pointer.
 *
 * mx_gemm_with_workspace - mx_gemm with caller-owned scratch memory.
 *   workspace        device memory, 16-byte aligned, owned by the caller; it
 *                    must stay untouched until the GEMM's work on `stream`
 *                    has finished. May be NULL when workspace_bytes == 0.
 *   workspace_bytes  its size. With less than mx_gemm_workspace_bytes the
 *                    GEMM runs whole tiles only: mx_gemm's result, never an
 *                    error.
 *   Everything else is exactly mx_gemm. The split adds one kernel launch on
 *   `stream`; both calls can be recorded into a CUDA graph.
 */
mx_status mx_gemm_workspace_bytes(int mode, const mx_operand* a, const mx_operand* b, size_t* bytes);
mx_status mx_gemm_with_workspace(int mode, const mx_operand* a, const mx_operand* b, void* c, int64_t ldc,
                                 void* workspace, size_t workspace_bytes, int* dev_status, void* stream);

/*
 * mx_gemm_static_workspace - mx_gemm_with_workspace for callers that must not
 * allocate device memory at all: not through cudaMalloc, not through a
 * framework's caching allocator, not by asking the caller for a buffer. Such
 * callers include code that runs inside a memory allocator's own callbacks
 * (allocating there would re-enter the allocator), runtimes that reserve all
 * of their device memory once at start-up and forbid allocation afterwards
 * (a later allocation can fail or fragment the reservation, and cudaFree
 * can synchronise the whole device), and plug-ins that receive only their
 * input and output buffers from a host application. (The pages have no
 * counterpart of this call: it is a property of this library's interface,
 * not of the method.)
 *
 * The split tail's scratch lives in one array of MX_STATIC_WORKSPACE_BYTES
 * bytes that the library declares in device memory. Each GPU that loads the
 * library's kernels holds that array until the process exits, whether or not
 * this call is used. The first call on a device looks up the array's device
 * address (a runtime query, no allocation) and caches it; make that first
 * call before any stream capture on the device.
 *
 *   Arguments, results, layouts and errors are exactly mx_gemm's, and the
 *   output equals mx_gemm_with_workspace's with a large enough caller
 *   workspace, bit for bit.
 *   A GEMM whose split tail would need more than MX_STATIC_WORKSPACE_BYTES
 *   (mx_gemm_workspace_bytes reports the need) is rejected with
 *   MX_ERR_UNSUPPORTED_SHAPE before anything is launched; on a GB300 (76 SM
 *   pairs) no GEMM needs more than 38 MiB.
 *   The array needs no clearing: a split GEMM writes every partial it reads
 *   back in the same call. But every call shares the one array and it keeps
 *   the last call's contents: two calls whose work overlaps on the GPU (on
 *   two streams, or two host threads) race on it and give wrong results.
 *   Order such calls on one stream, or use mx_gemm_with_workspace with a
 *   buffer per stream.
 */
#define MX_STATIC_WORKSPACE_BYTES (40u * 1024u * 1024u)
mx_status mx_gemm_static_workspace(int mode, const mx_operand* a, const mx_operand* b, void* c, int64_t ldc,
                                   int* dev_status, void* stream);

/* One GEMM of an mx_gemm_multi call: the arguments of mx_gemm. */
typedef struct mx_gemm_problem {
  mx_operand a;
  mx_operand b;
  void* c;          /* BF16 [a.rows, b.rows], row pitch ldc elements */
  int64_t ldc;
  int32_t mode;     /* MX_FPROP, MX_DGRAD or MX_WGRAD */
  int32_t reserved; /* must be 0 */
} mx_gemm_problem;

/*
 * mx_gemm_multi - up to MX_MAX_GEMM_MULTI independent dense GEMMs in one
 * launch, e.g. the dgrad and wgrad of one Linear layer's backward pass
 * ([DSV3] §8: both read the quantised dY, dgrad with W's column copy and
 * wgrad with X's; §10, the step data flow). One persistent grid walks the
 * tiles of all of them, so the GPU fills up across the GEMMs' last partial
 * rounds and pays one launch. Each output equals mx_gemm's for that problem
 * up to FP32 summation order (whole tiles; no split tail), within the same
 * bound; results are bit-identical from call to call.
 *
 *   problems  host array of n descriptors (read before return).
 *   n         0 .. MX_MAX_GEMM_MULTI.
 *   Requirements per problem are mx_gemm's; any violation fails the whole
 *   call before anything is launched (mx_last_error names the problem).
 *   No output may overlap another output or any operand: the GEMMs run
 *   concurrently.
 */
#define MX_MAX_GEMM_MULTI 4
mx_status mx_gemm_multi(const mx_gemm_problem* problems, int n, int* dev_status, void* stream);

/*
 * mx_grouped_gemm - per-expert block-scaled GEMMs over contiguous token ranges
 * ([DSV3] §5.2 routed experts and §13.4 low_precision_grouped_matmul with
 * group_list; [TT] npu_grouped_matmul). group_offsets is the int64 device array
 * described for mx_quantize. Empty and uneven groups are allowed ([DSV3] §16.3);
 * 1 <= n_groups <= MX_MAX_GROUPS.
 *
 *   MX_FPROP / MX_DGRAD (rows ragged): a = [M_total, K] row copy whose rows are
 *     grouped by expert; b = stacked per-expert copies: expert e's rows start at
 *     b->data + e*b->rows*ld and its scales at b->scale + e*mx_scale_bytes(b->rows, K);
 *     c = [M_total, N] (pitch ldc). Rows of group e use expert e's weights.
 *   MX_WGRAD (contraction ragged): a = grouped column copy of dY [N, cap],
 *     b = grouped column copy of X [Kout, cap] (both from mx_quantize with the
 *     same offsets and cap = a->k = b->k); c = [n_groups, N, Kout] with row
 *     pitch ldc and expert stride N*ldc. An empty group writes exact zeros.
 */
mx_status mx_grouped_gemm(int mode, const mx_operand* a, const mx_operand* b,
                          const int64_t* group_offsets, int n_groups, void* c, int64_t ldc,
                          int* dev_status, void* stream);

/*
 * Variant recipe: DeepSeek-V3 blockwise FP8 ("浮点格式、数值稳定性与混合精度"
 * §七.2-§七.3). E4M3 data with one FP32 multiplier per block, s = 448 / amax
 * (an all-zero block takes s = 1), element = E4M3(s * x) with the product
 * rounded to FP32 and then to E4M3 (nearest, ties to even, saturating).
 * Blocks holding Inf or NaN are outside this recipe.
 *
 * mx_quantize_fp8_blockwise - x BF16 [rows, cols] (pitch ldx, a multiple of 8;
 * 16-byte aligned), cols % 128 == 0; data E4M3 [rows, cols] (pitch cols).
 *   block = 1:   1 x 128 activation blocks; scale FP32 [cols/128][rows] (one
 *                row of multipliers per 128-column block, transposed so a
 *                GEMM tile's rows are contiguous).
 *   block = 128: 128 x 128 weight blocks (the last row block may be short);
 *                scale FP32 [ceil(rows/128)][cols/128].
 */
mx_status mx_quantize_fp8_blockwise(const void* x, int64_t rows, int64_t cols, int64_t ldx, int block, void* data,
                                    float* scale, int* dev_status, void* stream);

/*
 * mx_gemm_fp8_blockwise - C[M, N] = sum over 128-K blocks kb of
 * (A_kb . B_kb^T) / (a_scale[kb][m] * b_scale[n/128][kb]): each block's partial
 * sum is promoted to FP32 with its two multipliers (same page, §七.3). a_data
 * E4M3 [M, K] from block = 1, b_data E4M3 [N, K] from block = 128 (both dense,
 * pitch K, 16-byte aligned), K % 128 == 0; C BF16 [M, N] pitch ldc, round to
 * nearest even. Errors as mx_gemm.
 */
mx_status mx_gemm_fp8_blockwise(const void* a_data, const float* a_scale, int64_t M, const void* b_data,
                                const float* b_scale, int64_t N, int64_t K, void* c, int64_t ldc, int* dev_status,
                                void* stream);

/*
 * Variant recipe: current scaling with one FP32 scale per tensor or per
 * leading group ("DeepSeek-V3 16B FSDP2 MXFP8/HiF8 训练设计" §3: HiF8 current
 * scaling takes an FP32 scale from the current tensor's amax, a scalar for a
 * dense tensor and one per leading group for a grouped one; §3.2: scale =
 * valid(amax) ? amax / format_max : 1.0 in FP32, dense tensors per tensor,
 * 3-D grouped weights per leading group; §8.2: activations and gradients take
 * amax and scale at every quantisation, weights after the optimizer step).
 * Here the data are E4M3 codes, so format_max is normally 448 (E4M3's largest
 * value); the HiF8 dtype itself is not built. An element's code is
 * E4M3(fl32(x / scale)): the quotient rounded to FP32, then to nearest E4M3,
 * ties to even, saturating at 448 (NaN keeps its sign, +-Inf gives +-448).
 * A valid amax is finite and above zero; otherwise the scale is 1.
 *
 * mx_current_amax - amax[b] = max |x| over matrix b of a BF16 stack
 *   ([batch][rows, cols], row pitch ldx, matrix stride x_batch_stride
 *   elements; cols % 32 == 0; x 16-byte aligned, ldx and the stride multiples
 *   of 8). amax: FP32 device array of batch entries, written (NaN if a matrix
 *   holds NaN, +Inf if it holds an infinity, 0 for an empty matrix). The
 *   values can be combined (e.g. a maximum across ranks) before
 *   mx_quantize_current reads them.
 *
 * mx_quantize_current - quantise with scale[b] = amax[b] / format_max (FP32;
 *   1 for an invalid amax), written to scale (FP32 device array of batch).
 *   The scale does not depend on the direction, so the two copies hold the
 *   same codes in two layouts, each K-major for the GEMMs below:
 *   row copy (MX_ROWWISE/BOTH): row_data [batch][rows][cols];
 *   column copy (MX_COLWISE/BOTH): col_data [batch][cols][rows] (rows % 32 ==
 *     0), or, with group offsets (batch 1, the int64 device offsets of
 *     mx_quantize, 1 <= n_groups <= MX_MAX_GROUPS), [cols][col_capacity] with
 *     group e's rows at columns poff[e] .. and zero codes in each segment's
 *     padding to a multiple of 128 (the layout of mx_quantize's grouped column
 *     copy). Outputs 16-byte aligned; errors as mx_quantize.
 *
 * mx_gemm_current / mx_grouped_gemm_current - mx_gemm / mx_grouped_gemm on
 *   such operands: each mx_operand's `scale` is the FP32 scale array written
 *   by mx_quantize_current (4-byte aligned): one value for an activation, a
 *   gradient or a dense weight; one per expert for stacked expert weights
 *   (b of the rows-ragged fprop and dgrad). C = (A_codes . B_codes^T) * s_a *
 *   s_b with FP32 accumulation, the product of the two scales applied to the
 *   FP32 accumulator once, then BF16 round-to-nearest-even. Modes, layouts,
 *   groups and errors as mx_gemm / mx_grouped_gemm (wgrad: a and b are the
 *   grouped column copies of dY and X, each with its one scale).
 */
mx_status mx_current_amax(const void* x, int64_t batch, int64_t rows, int64_t cols, int64_t ldx,
                          int64_t x_batch_stride, float* amax, int* dev_status, void* stream);
mx_status mx_quantize_current(const void* x, int64_t batch, int64_t rows, int64_t cols, int64_t ldx,
                              int64_t x_batch_stride, int axis, const float* amax, float format_max, void* row_data,
                              void* col_data, float* scale, const int64_t* group_offsets, int n_groups,
                              int64_t col_capacity, int* dev_status, void* stream);
mx_status mx_gemm_current(int mode, const mx_operand* a, const mx_operand* b, void* c, int64_t ldc, int* dev_status,
                          void* stream);
mx_status mx_grouped_gemm_current(int mode, const mx_operand* a, const mx_operand* b, const int64_t* group_offsets,
                                  int n_groups, void* c, int64_t ldc, int* dev_status, void* stream);

/*
 * mx_gemm_current_multi - up to MX_MAX_GEMM_MULTI independent tensor-scaled
 * dense GEMMs (each as mx_gemm_current, operands from mx_quantize_current) in
 * one launch, e.g. a layer's dgrad and wgrad (the step data flow of
 * "DeepSeek-V3 16B FSDP2 MXFP8/HiF8 训练设计" §10 with the current-scaling
 * recipe of §3.2 / §8.2). Problem descriptors, requirements and errors as
 * mx_gemm_multi; every output equals mx_gemm_current's for that problem bit
 * for bit (the same whole tiles in the same order).
 */
mx_status mx_gemm_current_multi(const mx_gemm_problem* problems, int n, int* dev_status, void* stream);

/*
 * mx_grouped_gemm_swiglu - the routed experts' gate_up fprop with the grouped
 * SwiGLU fused into its epilogue ("DeepSeek-V3 16B FSDP2 MXFP8/HiF8 训练设计"
 * §5: gate_up_proj [E, 2F, H] and the grouped SwiGLU between gate_up and
 * down; §1: SwiGLU is not a low-precision operator, so it is evaluated in FP32
 * on the FP32 accumulators and rounded once to BF16).
 *
 *   a       row copy of the tokens [M_total, K], rows grouped by expert as in
 *           mx_grouped_gemm (MX_FPROP contract).
 *   b       stacked row copies of gate_up [E][2F][K]: rows [0, F) of each
 *           expert are its gate projection, rows [F, 2F) its up projection;
 *           2F must be a multiple of 256.
 *   c       BF16 [M_total, F], row pitch ldc: c[i, f] = silu(g) * u with
 *           g = (A . B_e^T)[i, f], u = (A . B_e^T)[i, F + f], e the expert of row
 *           i, silu(x) = x / (1 + exp(-x)).
 *   Groups (at most MX_MAX_GROUPS), validation, empty experts and errors as
 *   mx_grouped_gemm.
 */
mx_status mx_grouped_gemm_swiglu(const mx_operand* a, const mx_operand* b, const int64_t* group_offsets,
                                 int n_groups, void* c, int64_t ldc, int* dev_status, void* stream);

/*
 * mx_grouped_gemm_swiglu_quantize - mx_grouped_gemm_swiglu with its output
 * quantised in the same epilogue: instead of the BF16 [M_total, F] output it
 * writes that output's MX copies, byte for byte what mx_quantize(output,
 * MX_BOTH, group_offsets, col_capacity) would write from it (the output
 * values rounded to BF16 exactly as mx_grouped_gemm_swiglu stores them, then
 * the block rule of mx_quantize). These are the down projection's operands:
 * the row copy for its fprop, the per-expert column copy for its wgrad
 * ("DeepSeek-V3 16B FSDP2 MXFP8/HiF8 训练设计" §5 and §12.2: quantise by role
 * before the GEMMs that read the tensor).
 *
 *   a, b, group_offsets, n_groups   as mx_grouped_gemm_swiglu.
 *   row_data   E4M3 [M_total, F]; row_scale  mx_scale_bytes(M_total, F) bytes.
 *   col_data   E4M3 [F, col_capacity]: group e's rows at columns poff[e] ..,
 *              each segment zero-padded to a multiple of 128 rows (the layout
 *              of mx_quantize's grouped column copy); col_scale
 *              mx_scale_bytes(F, col_capacity) bytes. Columns past the last
 *              segment are not written.
 *   col_capacity  a positive multiple of 128, at least the sum over groups of
 *              their rows rounded up to 128 (mx_grouped_padded_rows); a
 *              smaller sum on the device is MX_ERR_DEVICE_CHECK in dev_status.
 *   All four outputs 16-byte aligned and owned by the caller. K = 0 zeroes all
 *   four buffers (silu(0) * 0 = 0). Errors otherwise as mx_grouped_gemm_swiglu.
 */
mx_status mx_grouped_gemm_swiglu_quantize(const mx_operand* a, const mx_operand* b, const int64_t* group_offsets,
                                          int n_groups, void* row_data, void* row_scale, void* col_data,
                                          void* col_scale, int64_t col_capacity, int* dev_status, void* stream);

/* Static description of a status code. */
const char* mx_status_string(mx_status s);

/* Message of the last MX_ERR_CUDA / validation failure on this host thread. */
const char* mx_last_error(void);

/* MXFP8_ABI_VERSION of the loaded library. */
int mx_abi_version(void);

/*
 * mx_selftest_wait_timeout - failure-reporting self test: launches one CTA
 * whose thread waits, through the same bounded mbarrier wait every kernel of
 * the library uses, on a barrier that nothing ever signals. When timeout_ns
 * expires the kernel writes MX_ERR_TIMEOUT to *dev_status and returns; the
 * context stays usable. dev_status must be a device int (0 before the call);
 * 0 < timeout_ns <= 10 s. Asynchronous on stream.
 *
 * (Every kernel's waits are bounded by MXFP8_WAIT_TIMEOUT_NS nanoseconds,
 * default 2 s, at least 1 ms; on expiry the kernel records MX_ERR_TIMEOUT,
 * lets its own copies and MMAs land, frees its tensor memory and returns.)
 */
mx_status mx_selftest_wait_timeout(uint64_t timeout_ns, int* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MXFP8_GB300_H */
