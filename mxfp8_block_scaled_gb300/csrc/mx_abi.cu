// mx_abi.cu - the C ABI (include/mxfp8.h): host-side validation, dispatch
// to the kernels on the caller's stream, status strings. No device memory is
// allocated here or anywhere else in the library.

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "mx_internal.h"
#include "mx_ptx.cuh"

namespace mx {

namespace {
thread_local char g_err[512] = "";

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The current device must be an sm_103 part (the kernels are built for sm_103a only).
mx_status check_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e, "cudaGetDevice");
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) {
    set_error("device %d is sm_%d%d; this library runs on sm_103 only", dev, major, minor);
    return MX_ERR_NO_DEVICE;
  }
  return MX_OK;
}

mx_status check_operand(const mx_operand* o, const char* name) {
  if (!o) {
    set_error("%s: null operand", name);
    return MX_ERR_INVALID_ARG;
  }
  if (o->rows < 0 || o->k < 0 || o->ld < 0 || o->reserved != 0) {
    set_error("%s: negative size or reserved field set", name);
    return MX_ERR_INVALID_ARG;
  }
  if (o->orient != MX_ROWWISE && o->orient != MX_COLWISE) {
    set_error("%s: orient must be MX_ROWWISE or MX_COLWISE", name);
    return MX_ERR_INVALID_ARG;
  }
  const int64_t ld = o->ld ? o->ld : o->k;
  if (ld < o->k) {
    set_error("%s: ld < k", name);
    return MX_ERR_INVALID_ARG;
  }
  if (o->k % 32 != 0) {
    set_error("%s: k = %lld is not a multiple of 32", name, static_cast<long long>(o->k));
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  if (o->rows > 0 && o->k > 0) {
    if (!o->data || !o->scale) {
      set_error("%s: null data or scale", name);
      return MX_ERR_INVALID_ARG;
    }
    if (!aligned16(o->data) || !aligned16(o->scale) || ld % 16 != 0) {
      set_error("%s: data/scale must be 16-byte aligned and ld a multiple of 16", name);
      return MX_ERR_ALIGNMENT;
    }
  }
  return MX_OK;
}

// fprop (row, row), dgrad (row of dY, col of W), wgrad (col of dY, col of X):
// the direction table of the design page, §8.
mx_status check_mode(int mode, const mx_operand* a, const mx_operand* b) {
  int want_a, want_b;
  switch (mode) {
    case MX_FPROP: want_a = MX_ROWWISE; want_b = MX_ROWWISE; break;
    case MX_DGRAD: want_a = MX_ROWWISE; want_b = MX_COLWISE; break;
    case MX_WGRAD: want_a = MX_COLWISE; want_b = MX_COLWISE; break;
    default:
      set_error("unknown GEMM mode %d", mode);
      return MX_ERR_INVALID_ARG;
  }
  if (a->orient != want_a || b->orient != want_b) {
    set_error("mode %d needs operand orientations (%d, %d), got (%d, %d)", mode, want_a, want_b, a->orient,
              b->orient);
    return MX_ERR_INVALID_ARG;
  }
  return MX_OK;
}

mx_status check_output(void* c, int64_t ldc, int64_t N, int64_t rows) {
  if (rows > 0 && N > 0) {
    if (!c) {
      set_error("null output");
      return MX_ERR_INVALID_ARG;
    }
    if (ldc < N) {
      set_error("ldc < N");
      return MX_ERR_INVALID_ARG;
    }
    if ((reinterpret_cast<uintptr_t>(c) & 1u) != 0) {
      set_error("output must be 2-byte aligned (BF16)");
      return MX_ERR_ALIGNMENT;
    }
  }
  return MX_OK;
}

mx_status zero_output(void* c, int64_t ldc, int64_t N, int64_t rows, cudaStream_t s) {
  if (rows == 0 || N == 0) return MX_OK;
  return cuda_status(cudaMemset2DAsync(c, static_cast<size_t>(ldc) * 2, 0, static_cast<size_t>(N) * 2,
                                       static_cast<size_t>(rows), s),
                     "cudaMemset2DAsync");
}
}  // namespace

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

mx_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return MX_OK;
  set_error("%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
  return MX_ERR_CUDA;
}

bool pdl_enabled() {
  static const bool on = [] {
    const char* s = std::getenv("MXFP8_PDL");
    return !(s && *s && std::atoi(s) == 0);
  }();
  return on;
}

uint64_t wait_timeout_ns() {
  // At least 1 ms: the drain after an abort waits for copies and MMAs already
  // in flight (they finish within microseconds) under the same bound.
  static uint64_t v = [] {
    const char* s = std::getenv("MXFP8_WAIT_TIMEOUT_NS");
    if (s && *s) {
      const unsigned long long x = std::strtoull(s, nullptr, 10);
      if (x > 0) return std::max<uint64_t>(static_cast<uint64_t>(x), 1000000ull);
    }
    return static_cast<uint64_t>(2000000000ull);
  }();
  return v;
}

int sm_count() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  std::lock_guard<std::mutex> lk(mu);
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 1;
  }
  return cache[dev];
}

}  // namespace mx

using namespace mx;

// Stacked dense quantisation with BF16 (elem 2) or FP32 (elem 4) input.
static mx_status quantize_stacked(const char* fn, int elem, const void* x, int64_t batch, int64_t rows, int64_t cols,
                                  int64_t ldx, int64_t x_batch_stride, int axis, void* row_data, void* row_scale,
                                  void* col_data, void* col_scale, int* dev_status, void* stream) {
  const int64_t align_elems = 16 / elem;  // elements per 16 bytes
  if (batch < 0 || x_batch_stride < 0) {
    set_error("%s: negative batch or stride", fn);
    return MX_ERR_INVALID_ARG;
  }
  if (batch > 1 && x_batch_stride < rows * ldx) {
    set_error("%s: x_batch_stride < rows * ldx", fn);
    return MX_ERR_INVALID_ARG;
  }
  if (batch > 1 && x_batch_stride % align_elems != 0) {
    set_error("%s: x_batch_stride must be a multiple of 16 bytes", fn);
    return MX_ERR_ALIGNMENT;
  }
  if (batch > 0x7FFFFFFFLL) {
    set_error("%s: batch must be < 2^31", fn);
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  // Per-matrix validation is the dense mx_quantize's; a zero-size problem is a no-op.
  if (batch == 0) {
    return (axis == MX_ROWWISE || axis == MX_COLWISE || axis == MX_BOTH) ? MX_OK : MX_ERR_INVALID_ARG;
  }
  if (axis != MX_ROWWISE && axis != MX_COLWISE && axis != MX_BOTH) {
    set_error("%s: axis must be MX_ROWWISE, MX_COLWISE or MX_BOTH", fn);
    return MX_ERR_INVALID_ARG;
  }
  if (rows < 0 || cols < 0 || ldx < cols) {
    set_error("%s: bad sizes", fn);
    return MX_ERR_INVALID_ARG;
  }
  if (rows > 0x7FFFFFFFLL) {
    set_error("%s: rows must be < 2^31", fn);
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  const bool do_row = (axis & MX_ROWWISE) != 0;
  const bool do_col = (axis & MX_COLWISE) != 0;
  if (cols % 32 != 0 || (do_col && rows % 32 != 0)) {
    set_error("%s: cols (and rows for the column copy) must be multiples of 32", fn);
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  if (rows == 0 || cols == 0) return MX_OK;
  if (!x || !aligned16(x) || ldx % align_elems != 0) {
    set_error("%s: x must be non-null and 16-byte aligned, rows 16-byte aligned (ldx)", fn);
    return x ? MX_ERR_ALIGNMENT : MX_ERR_INVALID_ARG;
  }
  if ((do_row && (!row_data || !row_scale)) || (do_col && (!col_data || !col_scale))) {
    set_error("%s: a requested output is null", fn);
    return MX_ERR_INVALID_ARG;
  }
  if ((do_row && (!aligned16(row_data) || !aligned16(row_scale))) ||
      (do_col && (!aligned16(col_data) || !aligned16(col_scale)))) {
    set_error("%s: outputs must be 16-byte aligned", fn);
    return MX_ERR_ALIGNMENT;
  }
  mx_status st = check_device();
  if (st != MX_OK) return st;
  QuantLaunch q;
  q.x = x;
  q.rows = rows;
  q.cols = cols;
  q.ldx = ldx;
  q.row_data = row_data;
  q.row_scale = row_scale;
  q.col_data = col_data;
  q.col_scale = col_scale;
  q.offsets = nullptr;
  q.n_groups = 0;
  q.col_pitch = rows;
  q.batch = batch;
  q.x_batch_stride = x_batch_stride;
  q.x_f32 = (elem == 4);
  q.dev_status = dev_status;
  return launch_quantize(q, do_row, do_col, static_cast<cudaStream_t>(stream));
}

// One thread waits, through the library's bounded wait, on an mbarrier that
// nothing ever arrives on; when the bound expires it reports MX_ERR_TIMEOUT
// the way every kernel of the library does.
__global__ void selftest_wait_kernel(uint64_t timeout_ns, int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, timeout_ns)) atomicExch(status, static_cast<int>(MX_ERR_TIMEOUT));
}

extern "C" {

int mx_abi_version(void) { return MXFP8_ABI_VERSION; }

mx_status mx_selftest_wait_timeout(uint64_t timeout_ns, int* dev_status, void* stream) {
  if (!dev_status || timeout_ns == 0 || timeout_ns > 10000000000ull) {
    set_error("mx_selftest_wait_timeout: dev_status must be non-null and 0 < timeout_ns <= 10 s");
    return MX_ERR_INVALID_ARG;
  }
  mx_status st = check_device();
  if (st != MX_OK) return st;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(timeout_ns, dev_status);
  return cuda_status(cudaGetLastError(), "mx_selftest_wait_timeout launch");
}

const char* mx_last_error(void) { return g_err; }

const char* mx_status_string(mx_status s) {
  switch (s) {
    case MX_OK: return "MX_OK";
    case MX_ERR_INVALID_ARG: return "MX_ERR_INVALID_ARG: invalid argument";
    case MX_ERR_UNSUPPORTED_SHAPE: return "MX_ERR_UNSUPPORTED_SHAPE: unsupported shape";
    case MX_ERR_ALIGNMENT: return "MX_ERR_ALIGNMENT: pointer or pitch not 16-byte aligned";
    case MX_ERR_CUDA: return "MX_ERR_CUDA: CUDA call failed";
    case MX_ERR_DEVICE_CHECK: return "MX_ERR_DEVICE_CHECK: device-side validation failed";
    case MX_ERR_TIMEOUT: return "MX_ERR_TIMEOUT: bounded device wait expired";
    case MX_ERR_NO_DEVICE: return "MX_ERR_NO_DEVICE: current device is not sm_103";
  }
  return "unknown mx_status";
}

size_t mx_scale_bytes(int64_t rows, int64_t k) {
  if (rows <= 0 || k <= 0) return 0;
  const int64_t kb = (k + 31) / 32;
  return static_cast<size_t>((rows + 127) / 128 * 128) * static_cast<size_t>((kb + 3) / 4 * 4);
}

int64_t mx_grouped_padded_rows(const int64_t* host_offsets, int n_groups) {
  if (!host_offsets || n_groups < 0 || host_offsets[0] != 0) return -1;
  int64_t total = 0;
  for (int e = 0; e < n_groups; ++e) {
    const int64_t m = host_offsets[e + 1] - host_offsets[e];
    if (m < 0) return -1;
    total += (m + 127) / 128 * 128;
  }
  return total;
}

mx_status mx_quantize(const void* x, int64_t rows, int64_t cols, int64_t ldx, int axis, void* row_data,
                      void* row_scale, void* col_data, void* col_scale, const int64_t* group_offsets,
                      int n_groups, int64_t col_capacity, int* dev_status, void* stream) {
  if (axis != MX_ROWWISE && axis != MX_COLWISE && axis != MX_BOTH) {
    set_error("mx_quantize: axis must be MX_ROWWISE, MX_COLWISE or MX_BOTH");
    return MX_ERR_INVALID_ARG;
  }
  if (rows < 0 || cols < 0 || ldx < cols) {
    set_error("mx_quantize: bad sizes rows=%lld cols=%lld ldx=%lld", static_cast<long long>(rows),
              static_cast<long long>(cols), static_cast<long long>(ldx));
    return MX_ERR_INVALID_ARG;
  }
  if (rows > 0x7FFFFFFFLL) {
    set_error("mx_quantize: rows must be < 2^31");
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  const bool do_row = (axis & MX_ROWWISE) != 0;
  const bool do_col = (axis & MX_COLWISE) != 0;
  const bool grouped = group_offsets != nullptr;
  if (cols % 32 != 0) {
    set_error("mx_quantize: cols = %lld is not a multiple of 32", static_cast<long long>(cols));
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  if (do_col && !grouped && rows % 32 != 0) {
    set_error("mx_quantize: dense column copy needs rows %% 32 == 0 (rows = %lld)", static_cast<long long>(rows));
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  if (grouped) {
    if (!do_col) {
      set_error("mx_quantize: group offsets only apply to the column copy");
      return MX_ERR_INVALID_ARG;
    }
    if (n_groups < 1) {
      set_error("mx_quantize: n_groups must be >= 1");
      return MX_ERR_INVALID_ARG;
    }
    if (n_groups > MX_MAX_GROUPS) {
      set_error("mx_quantize: n_groups = %d is above MX_MAX_GROUPS (%d)", n_groups, MX_MAX_GROUPS);
      return MX_ERR_UNSUPPORTED_SHAPE;
    }
    if (col_capacity < 0 || col_capacity % 128 != 0) {
      set_error("mx_quantize: col_capacity must be a non-negative multiple of 128");
      return MX_ERR_UNSUPPORTED_SHAPE;
    }
  }
  if (rows == 0 || cols == 0) return MX_OK;
  if (!x || !aligned16(x) || ldx % 8 != 0) {
    set_error("mx_quantize: x must be non-null, 16-byte aligned, ldx a multiple of 8");
    return x ? MX_ERR_ALIGNMENT : MX_ERR_INVALID_ARG;
  }
  if (do_row && (!row_data || !row_scale)) {
    set_error("mx_quantize: row copy requested but row_data/row_scale is null");
    return MX_ERR_INVALID_ARG;
  }
  if (do_col && (!col_data || !col_scale)) {
    set_error("mx_quantize: column copy requested but col_data/col_scale is null");
    return MX_ERR_INVALID_ARG;
  }
  if ((do_row && (!aligned16(row_data) || !aligned16(row_scale))) ||
      (do_col && (!aligned16(col_data) || !aligned16(col_scale)))) {
    set_error("mx_quantize: outputs must be 16-byte aligned");
    return MX_ERR_ALIGNMENT;
  }
  if (grouped && col_capacity == 0) {
    set_error("mx_quantize: col_capacity is 0 but rows > 0");
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  mx_status st = check_device();
  if (st != MX_OK) return st;
  QuantLaunch q;
  q.x = x;
  q.rows = rows;
  q.cols = cols;
  q.ldx = ldx;
  q.row_data = row_data;
  q.row_scale = row_scale;
  q.col_data = col_data;
  q.col_scale = col_scale;
  q.offsets = group_offsets;
  q.n_groups = n_groups;
  q.col_pitch = grouped ? col_capacity : rows;
  q.batch = 1;
  q.x_batch_stride = 0;
  q.dev_status = dev_status;
  return launch_quantize(q, do_row, do_col, static_cast<cudaStream_t>(stream));
}

mx_status mx_quantize_batched(const void* x, int64_t batch, int64_t rows, int64_t cols, int64_t ldx,
                              int64_t x_batch_stride, int axis, void* row_data, void* row_scale, void* col_data,
                              void* col_scale, int* dev_status, void* stream) {
  return quantize_stacked("mx_quantize_batched", 2, x, batch, rows, cols, ldx, x_batch_stride, axis, row_data,
                          row_scale, col_data, col_scale, dev_status, stream);
}

mx_status mx_quantize_f32(const float* x, int64_t batch, int64_t rows, int64_t cols, int64_t ldx,
                          int64_t x_batch_stride, int axis, void* row_data, void* row_scale, void* col_data,
                          void* col_scale, int* dev_status, void* stream) {
  return quantize_stacked("mx_quantize_f32", 4, x, batch, rows, cols, ldx, x_batch_stride, axis, row_data,
                          row_scale, col_data, col_scale, dev_status, stream);
}

mx_status mx_quantize_multi(const mx_quant_tensor* tensors, int n, int axis, int* dev_status, void* stream) {
  if (axis != MX_ROWWISE && axis != MX_COLWISE && axis != MX_BOTH) {
    set_error("mx_quantize_multi: axis must be MX_ROWWISE, MX_COLWISE or MX_BOTH");
    return MX_ERR_INVALID_ARG;
  }
  if (n < 0 || n > MX_MAX_MULTI) {
    set_error("mx_quantize_multi: n = %d is outside 0 .. %d", n, MX_MAX_MULTI);
    return MX_ERR_INVALID_ARG;
  }
  if (n == 0) return MX_OK;
  if (!tensors) {
    set_error("mx_quantize_multi: tensors is null");
    return MX_ERR_INVALID_ARG;
  }
  const bool do_row = (axis & MX_ROWWISE) != 0;
  const bool do_col = (axis & MX_COLWISE) != 0;
  QuantLaunch qs[MX_MAX_MULTI];
  int m = 0;
  // Every matrix is checked before anything is launched.
  for (int i = 0; i < n; ++i) {
    const mx_quant_tensor& t = tensors[i];
    if (t.rows < 0 || t.cols < 0 || t.ldx < t.cols) {
      set_error("mx_quantize_multi: tensor %d: bad sizes rows=%lld cols=%lld ldx=%lld", i,
                static_cast<long long>(t.rows), static_cast<long long>(t.cols), static_cast<long long>(t.ldx));
      return MX_ERR_INVALID_ARG;
    }
    if (t.rows > 0x7FFFFFFFLL) {
      set_error("mx_quantize_multi: tensor %d: rows must be < 2^31", i);
      return MX_ERR_UNSUPPORTED_SHAPE;
    }
    if (t.cols % 32 != 0 || (do_col && t.rows % 32 != 0)) {
      set_error("mx_quantize_multi: tensor %d: cols (and rows for the column copy) must be multiples of 32", i);
      return MX_ERR_UNSUPPORTED_SHAPE;
    }
    if (t.rows == 0 || t.cols == 0) continue;
    if (!t.x || !aligned16(t.x) || t.ldx % 8 != 0) {
      set_error("mx_quantize_multi: tensor %d: x must be non-null, 16-byte aligned, ldx a multiple of 8", i);
      return t.x ? MX_ERR_ALIGNMENT : MX_ERR_INVALID_ARG;
    }
    if ((do_row && (!t.row_data || !t.row_scale)) || (do_col && (!t.col_data || !t.col_scale))) {
      set_error("mx_quantize_multi: tensor %d: a requested output is null", i);
      return MX_ERR_INVALID_ARG;
    }
    if ((do_row && (!aligned16(t.row_data) || !aligned16(t.row_scale))) ||
        (do_col && (!aligned16(t.col_data) || !aligned16(t.col_scale)))) {
      set_error("mx_quantize_multi: tensor %d: outputs must be 16-byte aligned", i);
      return MX_ERR_ALIGNMENT;
    }
    QuantLaunch& q = qs[m++];
    q = QuantLaunch();
    q.x = t.x;
    q.rows = t.rows;
    q.cols = t.cols;
    q.ldx = t.ldx;
    q.row_data = t.row_data;
    q.row_scale = t.row_scale;
    q.col_data = t.col_data;
    q.col_scale = t.col_scale;
    q.offsets = nullptr;
    q.n_groups = 0;
    q.col_pitch = t.rows;
    q.batch = 1;
    q.x_batch_stride = 0;
    q.dev_status = dev_status;
  }
  if (m == 0) return MX_OK;
  mx_status st = check_device();
  if (st != MX_OK) return st;
  return launch_quantize_multi(qs, m, do_row, do_col, static_cast<cudaStream_t>(stream));
}

// Dense GEMM checks shared by the entry points; fills L (dense, no workspace).
static mx_status dense_gemm_setup(const char* fn, int mode, const mx_operand* a, const mx_operand* b, void* c,
                                  int64_t ldc, int* dev_status, bool check_c, GemmLaunch* L) {
  mx_status st = check_operand(a, "a");
  if (st != MX_OK) return st;
  st = check_operand(b, "b");
  if (st != MX_OK) return st;
  st = check_mode(mode, a, b);
  if (st != MX_OK) return st;
  if (a->k != b->k) {
    set_error("%s: a.k (%lld) != b.k (%lld)", fn, static_cast<long long>(a->k), static_cast<long long>(b->k));
    return MX_ERR_INVALID_ARG;
  }
  if (a->rows > 0x7FFFFFFFLL || b->rows > 0x7FFFFFFFLL || a->k > 0x7FFFFFFFLL) {
    set_error("%s: sizes must be < 2^31", fn);
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  if (check_c) {
    st = check_output(c, ldc, b->rows, a->rows);
    if (st != MX_OK) return st;
  }
  L->kind = GEMM_DENSE;
  L->a_data = a->data;
  L->a_scale = a->scale;
  L->a_ld = a->ld ? a->ld : a->k;
  L->b_data = b->data;
  L->b_scale = b->scale;
  L->b_ld = b->ld ? b->ld : b->k;
  L->M = a->rows;
  L->N = b->rows;
  L->K = a->k;
  L->b_rows_total = b->rows;
  L->c = c;
  L->ldc = ldc;
  L->offsets = nullptr;
  L->n_groups = 0;
  L->dev_status = dev_status;
  return MX_OK;
}

static mx_status dense_gemm_run(GemmLaunch& L, void* stream) {
  if (L.M == 0 || L.N == 0) return MX_OK;
  mx_status st = check_device();
  if (st != MX_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (L.K == 0) return zero_output(L.c, L.ldc, L.N, L.M, s);
  return launch_gemm(L, s);
}

mx_status mx_gemm(int mode, const mx_operand* a, const mx_operand* b, void* c, int64_t ldc, int* dev_status,
                  void* stream) {
  GemmLaunch L;
  mx_status st = dense_gemm_setup("mx_gemm", mode, a, b, c, ldc, dev_status, true, &L);
  if (st != MX_OK) return st;
  return dense_gemm_run(L, stream);
}

mx_status mx_gemm_workspace_bytes(int mode, const mx_operand* a, const mx_operand* b, size_t* bytes) {
  if (!bytes) {
    set_error("mx_gemm_workspace_bytes: bytes is null");
    return MX_ERR_INVALID_ARG;
  }
  *bytes = 0;
  GemmLaunch L;
  mx_status st = dense_gemm_setup("mx_gemm_workspace_bytes", mode, a, b, nullptr, 0, nullptr, false, &L);
  if (st != MX_OK) return st;
  if (L.M == 0 || L.N == 0 || L.K == 0) return MX_OK;
  st = check_device();
  if (st != MX_OK) return st;
  *bytes = gemm_workspace_bytes(L);
  return MX_OK;
}

mx_status mx_gemm_with_workspace(int mode, const mx_operand* a, const mx_operand* b, void* c, int64_t ldc,
                                 void* workspace, size_t workspace_bytes, int* dev_status, void* stream) {
  GemmLaunch L;
  mx_status st = dense_gemm_setup("mx_gemm_with_workspace", mode, a, b, c, ldc, dev_status, true, &L);
  if (st != MX_OK) return st;
  if (workspace_bytes > 0 && (!workspace || !aligned16(workspace))) {
    set_error("mx_gemm_with_workspace: workspace must be non-null and 16-byte aligned when workspace_bytes > 0");
    return workspace ? MX_ERR_ALIGNMENT : MX_ERR_INVALID_ARG;
  }
  L.ws = workspace_bytes > 0 ? workspace : nullptr;
  L.ws_bytes = workspace_bytes;
  return dense_gemm_run(L, stream);
}

mx_status mx_gemm_static_workspace(int mode, const mx_operand* a, const mx_operand* b, void* c, int64_t ldc,
                                   int* dev_status, void* stream) {
  GemmLaunch L;
  mx_status st = dense_gemm_setup("mx_gemm_static_workspace", mode, a, b, c, ldc, dev_status, true, &L);
  if (st != MX_OK) return st;
  if (L.M == 0 || L.N == 0) return MX_OK;
  st = check_device();
  if (st != MX_OK) return st;
  if (L.K > 0) {
    const size_t need = gemm_workspace_bytes(L);
    if (need > MX_STATIC_WORKSPACE_BYTES) {
      set_error("mx_gemm_static_workspace: this GEMM needs %zu bytes of scratch, more than the %zu bytes of the "
                "static workspace; use mx_gemm_with_workspace with a caller buffer",
                need, static_cast<size_t>(MX_STATIC_WORKSPACE_BYTES));
      return MX_ERR_UNSUPPORTED_SHAPE;
    }
    if (need > 0) {
      st = static_workspace(&L.ws, &L.ws_bytes);
      if (st != MX_OK) return st;
    }
  }
  return dense_gemm_run(L, stream);
}

mx_status mx_gemm_multi(const mx_gemm_problem* problems, int n, int* dev_status, void* stream) {
  if (n < 0 || n > MX_MAX_GEMM_MULTI) {
    set_error("mx_gemm_multi: n = %d is outside 0 .. %d", n, MX_MAX_GEMM_MULTI);
    return MX_ERR_INVALID_ARG;
  }
  if (n == 0) return MX_OK;
  if (!problems) {
    set_error("mx_gemm_multi: problems is null");
    return MX_ERR_INVALID_ARG;
  }
  GemmLaunch Ls[MX_MAX_GEMM_MULTI];
  bool any = false;
  for (int i = 0; i < n; ++i) {
    const mx_gemm_problem& pr = problems[i];
    if (pr.reserved != 0) {
      set_error("mx_gemm_multi: problem %d: reserved must be 0", i);
      return MX_ERR_INVALID_ARG;
    }
    mx_status st = dense_gemm_setup("mx_gemm_multi", pr.mode, &pr.a, &pr.b, pr.c, pr.ldc, dev_status, true, &Ls[i]);
    if (st != MX_OK) {
      char msg[512];
      std::snprintf(msg, sizeof(msg), "%s", mx_last_error());
      set_error("problem %d: %s", i, msg);
      return st;
    }
    if (Ls[i].M > 0 && Ls[i].N > 0) any = true;
  }
  if (!any) return MX_OK;
  mx_status st = check_device();
  if (st != MX_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // K = 0: C = 0, no tensor-core work.
  GemmLaunch live[MX_MAX_GEMM_MULTI];
  int m = 0;
  for (int i = 0; i < n; ++i) {
    if (Ls[i].M == 0 || Ls[i].N == 0) continue;
    if (Ls[i].K == 0) {
      st = zero_output(Ls[i].c, Ls[i].ldc, Ls[i].N, Ls[i].M, s);
      if (st != MX_OK) return st;
      continue;
    }
    live[m++] = Ls[i];
  }
  return m ? launch_gemm_multi(live, m, s) : MX_OK;
}

static mx_status current_input_check(const char* fn, const void* x, int64_t batch, int64_t rows, int64_t cols,
                                     int64_t ldx, int64_t x_batch_stride) {
  if (batch < 0 || rows < 0 || cols < 0 || ldx < cols || x_batch_stride < 0) {
    set_error("%s: bad sizes", fn);
    return MX_ERR_INVALID_ARG;
  }
  if (batch > 0x7FFFFFFFLL || rows > 0x7FFFFFFFLL) {
    set_error("%s: batch and rows must be < 2^31", fn);
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  if (batch > 1 && x_batch_stride < rows * ldx) {
    set_error("%s: x_batch_stride < rows * ldx", fn);
    return MX_ERR_INVALID_ARG;
  }
  if (cols % 32 != 0) {
    set_error("%s: cols = %lld is not a multiple of 32", fn, static_cast<long long>(cols));
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  if (batch > 0 && rows > 0 && cols > 0) {
    if (!x) {
      set_error("%s: x is null", fn);
      return MX_ERR_INVALID_ARG;
    }
    if (!aligned16(x) || ldx % 8 != 0 || (batch > 1 && x_batch_stride % 8 != 0)) {
      set_error("%s: x must be 16-byte aligned with ldx and x_batch_stride multiples of 8", fn);
      return MX_ERR_ALIGNMENT;
    }
  }
  return MX_OK;
}

mx_status mx_current_amax(const void* x, int64_t batch, int64_t rows, int64_t cols, int64_t ldx,
                          int64_t x_batch_stride, float* amax, int* dev_status, void* stream) {
  (void)dev_status;
  mx_status st = current_input_check("mx_current_amax", x, batch, rows, cols, ldx, x_batch_stride);
  if (st != MX_OK) return st;
  if (batch == 0) return MX_OK;
  if (!amax || (reinterpret_cast<uintptr_t>(amax) & 3u) != 0) {
    set_error("mx_current_amax: amax must be a non-null, 4-byte aligned device array of batch floats");
    return amax ? MX_ERR_ALIGNMENT : MX_ERR_INVALID_ARG;
  }
  st = check_device();
  if (st != MX_OK) return st;
  QuantLaunch q{};
  q.x = x;
  q.rows = rows;
  q.cols = cols;
  q.ldx = ldx;
  q.batch = batch;
  q.x_batch_stride = x_batch_stride;
  return launch_current_amax(q, amax, static_cast<cudaStream_t>(stream));
}

mx_status mx_quantize_current(const void* x, int64_t batch, int64_t rows, int64_t cols, int64_t ldx,
                              int64_t x_batch_stride, int axis, const float* amax, float format_max, void* row_data,
                              void* col_data, float* scale, const int64_t* group_offsets, int n_groups,
                              int64_t col_capacity, int* dev_status, void* stream) {
  const char* fn = "mx_quantize_current";
  mx_status st = current_input_check(fn, x, batch, rows, cols, ldx, x_batch_stride);
  if (st != MX_OK) return st;
  if (axis != MX_ROWWISE && axis != MX_COLWISE && axis != MX_BOTH) {
    set_error("%s: axis must be MX_ROWWISE, MX_COLWISE or MX_BOTH", fn);
    return MX_ERR_INVALID_ARG;
  }
  if (!(format_max > 0.0f) || !(format_max <= 3.402823466e38f)) {
    set_error("%s: format_max must be finite and above zero", fn);
    return MX_ERR_INVALID_ARG;
  }
  const bool do_row = (axis & MX_ROWWISE) != 0;
  const bool do_col = (axis & MX_COLWISE) != 0;
  const bool grouped = group_offsets != nullptr;
  if (grouped) {
    if (!do_col || batch != 1 || n_groups < 1) {
      set_error("%s: group offsets apply to the column copy of one matrix, with n_groups >= 1", fn);
      return MX_ERR_INVALID_ARG;
    }
    if (n_groups > MX_MAX_GROUPS) {
      set_error("%s: n_groups = %d is above MX_MAX_GROUPS (%d)", fn, n_groups, MX_MAX_GROUPS);
      return MX_ERR_UNSUPPORTED_SHAPE;
    }
    if (col_capacity < 0 || col_capacity % 128 != 0) {
      set_error("%s: col_capacity must be a non-negative multiple of 128", fn);
      return MX_ERR_UNSUPPORTED_SHAPE;
    }
  } else if (do_col && rows % 32 != 0) {
    set_error("%s: the column copy needs rows %% 32 == 0", fn);
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  if (batch == 0) return MX_OK;
  if (!amax || !scale || (reinterpret_cast<uintptr_t>(amax) & 3u) || (reinterpret_cast<uintptr_t>(scale) & 3u)) {
    set_error("%s: amax and scale must be non-null, 4-byte aligned device arrays of batch floats", fn);
    return (amax && scale) ? MX_ERR_ALIGNMENT : MX_ERR_INVALID_ARG;
  }
  if (rows > 0 && cols > 0) {
    if ((do_row && !row_data) || (do_col && !col_data)) {
      set_error("%s: a requested output is null", fn);
      return MX_ERR_INVALID_ARG;
    }
    if ((do_row && !aligned16(row_data)) || (do_col && !aligned16(col_data))) {
      set_error("%s: outputs must be 16-byte aligned", fn);
      return MX_ERR_ALIGNMENT;
    }
    if (grouped && col_capacity == 0) {
      set_error("%s: col_capacity is 0 but rows > 0", fn);
      return MX_ERR_UNSUPPORTED_SHAPE;
    }
  }
  st = check_device();
  if (st != MX_OK) return st;
  QuantLaunch q{};
  q.x = x;
  q.rows = rows;
  q.cols = cols;
  q.ldx = ldx;
  q.row_data = row_data;
  q.col_data = col_data;
  q.offsets = group_offsets;
  q.n_groups = grouped ? n_groups : 0;
  q.col_pitch = grouped ? col_capacity : rows;
  q.batch = batch;
  q.x_batch_stride = x_batch_stride;
  q.dev_status = dev_status;
  return launch_quantize_current(q, amax, format_max, scale, do_row, do_col, static_cast<cudaStream_t>(stream));
}

// Operands of the current-scaling GEMMs: E4M3 codes as for mx_gemm, `scale`
// an FP32 device array (one scale, or one per expert for stacked weights).
static mx_status check_current_operand(const mx_operand* o, const char* name) {
  if (!o) {
    set_error("%s: null operand", name);
    return MX_ERR_INVALID_ARG;
  }
  mx_operand m = *o;
  const void* sc = m.scale;
  m.scale = m.data;  // the E8M0 checks do not apply to an FP32 scale
  mx_status st = check_operand(&m, name);
  if (st != MX_OK) return st;
  if (o->rows > 0 && o->k > 0) {
    if (!sc) {
      set_error("%s: null scale", name);
      return MX_ERR_INVALID_ARG;
    }
    if ((reinterpret_cast<uintptr_t>(sc) & 3u) != 0) {
      set_error("%s: the FP32 scale must be 4-byte aligned", name);
      return MX_ERR_ALIGNMENT;
    }
  }
  return MX_OK;
}

// Host checks and launch description of one tensor-scaled dense GEMM (shared
// by mx_gemm_current and mx_gemm_current_multi). L->M == 0 or L->N == 0:
// nothing to do; L->K == 0: the output is zeroed by the caller.
static mx_status current_gemm_setup(const char* fn, int mode, const mx_operand* a, const mx_operand* b, void* c,
                             int64_t ldc, int* dev_status, GemmLaunch* L) {
  mx_status st = check_current_operand(a, "a");
  if (st != MX_OK) return st;
  st = check_current_operand(b, "b");
  if (st != MX_OK) return st;
  st = check_mode(mode, a, b);
  if (st != MX_OK) return st;
  if (a->k != b->k) {
    set_error("%s: a.k != b.k", fn);
    return MX_ERR_INVALID_ARG;
  }
  if (a->rows > 0x7FFFFFFFLL || b->rows > 0x7FFFFFFFLL || a->k > 0x7FFFFFFFLL) {
    set_error("%s: sizes must be < 2^31", fn);
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  st = check_output(c, ldc, b->rows, a->rows);
  if (st != MX_OK) return st;
  L->kind = GEMM_DENSE;
  L->a_data = a->data;
  L->a_scale = a->scale;
  L->a_ld = a->ld ? a->ld : a->k;
  L->b_data = b->data;
  L->b_scale = b->scale;
  L->b_ld = b->ld ? b->ld : b->k;
  L->M = a->rows;
  L->N = b->rows;
  L->K = a->k;
  L->b_rows_total = b->rows;
  L->c = c;
  L->ldc = ldc;
  L->offsets = nullptr;
  L->n_groups = 0;
  L->dev_status = dev_status;
  L->tensor_scaled = true;
  return MX_OK;
}

mx_status mx_gemm_current(int mode, const mx_operand* a, const mx_operand* b, void* c, int64_t ldc, int* dev_status,
                          void* stream) {
  GemmLaunch L;
  mx_status st = current_gemm_setup("mx_gemm_current", mode, a, b, c, ldc, dev_status, &L);
  if (st != MX_OK) return st;
  if (L.M == 0 || L.N == 0) return MX_OK;
  st = check_device();
  if (st != MX_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (L.K == 0) return zero_output(c, ldc, L.N, L.M, s);
  return launch_gemm(L, s);
}

mx_status mx_gemm_current_multi(const mx_gemm_problem* problems, int n, int* dev_status, void* stream) {
  if (n < 0 || n > MX_MAX_GEMM_MULTI) {
    set_error("mx_gemm_current_multi: n = %d is outside 0 .. %d", n, MX_MAX_GEMM_MULTI);
    return MX_ERR_INVALID_ARG;
  }
  if (n == 0) return MX_OK;
  if (!problems) {
    set_error("mx_gemm_current_multi: problems is null");
    return MX_ERR_INVALID_ARG;
  }
  GemmLaunch Ls[MX_MAX_GEMM_MULTI];
  bool any = false;
  for (int i = 0; i < n; ++i) {
    const mx_gemm_problem& pr = problems[i];
    if (pr.reserved != 0) {
      set_error("mx_gemm_current_multi: problem %d: reserved must be 0", i);
      return MX_ERR_INVALID_ARG;
    }
    mx_status st = current_gemm_setup("mx_gemm_current_multi", pr.mode, &pr.a, &pr.b, pr.c, pr.ldc, dev_status, &Ls[i]);
    if (st != MX_OK) {
      char msg[512];
      std::snprintf(msg, sizeof(msg), "%s", mx_last_error());
      set_error("problem %d: %s", i, msg);
      return st;
    }
    if (Ls[i].M > 0 && Ls[i].N > 0) any = true;
  }
  if (!any) return MX_OK;
  mx_status st = check_device();
  if (st != MX_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  GemmLaunch live[MX_MAX_GEMM_MULTI];
  int m = 0;
  for (int i = 0; i < n; ++i) {
    if (Ls[i].M == 0 || Ls[i].N == 0) continue;
    if (Ls[i].K == 0) {
      st = zero_output(Ls[i].c, Ls[i].ldc, Ls[i].N, Ls[i].M, s);
      if (st != MX_OK) return st;
      continue;
    }
    live[m++] = Ls[i];
  }
  return m ? launch_gemm_multi(live, m, s) : MX_OK;
}

mx_status mx_grouped_gemm_current(int mode, const mx_operand* a, const mx_operand* b, const int64_t* group_offsets,
                                  int n_groups, void* c, int64_t ldc, int* dev_status, void* stream) {
  const char* fn = "mx_grouped_gemm_current";
  mx_status st = check_current_operand(a, "a");
  if (st != MX_OK) return st;
  st = check_current_operand(b, "b");
  if (st != MX_OK) return st;
  st = check_mode(mode, a, b);
  if (st != MX_OK) return st;
  if (!group_offsets || n_groups < 1) {
    set_error("%s: group_offsets must be non-null and n_groups >= 1", fn);
    return MX_ERR_INVALID_ARG;
  }
  if (n_groups > MX_MAX_GROUPS) {
    set_error("%s: n_groups = %d is above MX_MAX_GROUPS (%d)", fn, n_groups, MX_MAX_GROUPS);
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  if (a->k != b->k) {
    set_error("%s: a.k != b.k", fn);
    return MX_ERR_INVALID_ARG;
  }
  if (a->rows > 0x7FFFFFFFLL || b->rows > 0x7FFFFFFFLL || a->k > 0x7FFFFFFFLL) {
    set_error("%s: sizes must be < 2^31", fn);
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  GemmLaunch L;
  L.a_data = a->data;
  L.a_scale = a->scale;
  L.a_ld = a->ld ? a->ld : a->k;
  L.b_data = b->data;
  L.b_scale = b->scale;
  L.b_ld = b->ld ? b->ld : b->k;
  L.K = a->k;
  L.c = c;
  L.ldc = ldc;
  L.offsets = group_offsets;
  L.n_groups = n_groups;
  L.dev_status = dev_status;
  L.tensor_scaled = true;
  if (mode == MX_WGRAD) {
    if (a->k % 128 != 0) {
      set_error("%s: wgrad capacity (a.k) must be a multiple of 128", fn);
      return MX_ERR_UNSUPPORTED_SHAPE;
    }
    st = check_output(c, ldc, b->rows, a->rows * static_cast<int64_t>(n_groups));
    if (st != MX_OK) return st;
    if (a->rows == 0 || b->rows == 0) return MX_OK;
    st = check_device();
    if (st != MX_OK) return st;
    if (a->k == 0) return zero_output(c, ldc, b->rows, a->rows * static_cast<int64_t>(n_groups), s);
    L.kind = GEMM_GROUPED_K;
    L.M = a->rows;
    L.N = b->rows;
    L.b_rows_total = b->rows;
  } else {
    st = check_output(c, ldc, b->rows, a->rows);
    if (st != MX_OK) return st;
    if (a->rows == 0 || b->rows == 0) return MX_OK;
    st = check_device();
    if (st != MX_OK) return st;
    if (a->k == 0) return zero_output(c, ldc, b->rows, a->rows, s);
    L.kind = GEMM_GROUPED_M;
    L.M = a->rows;
    L.N = b->rows;
    L.b_rows_total = b->rows * static_cast<int64_t>(n_groups);
  }
  return launch_gemm(L, s);
}

mx_status mx_quantize_fp8_blockwise(const void* x, int64_t rows, int64_t cols, int64_t ldx, int block, void* data,
                                    float* scale, int* dev_status, void* stream) {
  (void)dev_status;
  if (block != 1 && block != 128) {
    set_error("mx_quantize_fp8_blockwise: block must be 1 (1 x 128 blocks) or 128 (128 x 128 blocks)");
    return MX_ERR_INVALID_ARG;
  }
  if (rows < 0 || cols < 0 || ldx < cols) {
    set_error("mx_quantize_fp8_blockwise: bad sizes");
    return MX_ERR_INVALID_ARG;
  }
  if (cols % 128 != 0) {
    set_error("mx_quantize_fp8_blockwise: cols must be a multiple of 128");
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  if (rows == 0 || cols == 0) return MX_OK;
  if (!x || !data || !scale) {
    set_error("mx_quantize_fp8_blockwise: null pointer");
    return MX_ERR_INVALID_ARG;
  }
  if (!aligned16(x) || ldx % 8 != 0 || !aligned16(data) || (reinterpret_cast<uintptr_t>(scale) & 3u) != 0) {
    set_error("mx_quantize_fp8_blockwise: x and data must be 16-byte aligned, ldx a multiple of 8, scale 4-byte aligned");
    return MX_ERR_ALIGNMENT;
  }
  mx_status st = check_device();
  if (st != MX_OK) return st;
  return launch_quantize_blockwise(x, rows, cols, ldx, block, data, scale, static_cast<cudaStream_t>(stream));
}

mx_status mx_gemm_fp8_blockwise(const void* a_data, const float* a_scale, int64_t M, const void* b_data,
                                const float* b_scale, int64_t N, int64_t K, void* c, int64_t ldc, int* dev_status,
                                void* stream) {
  if (M < 0 || N < 0 || K < 0) {
    set_error("mx_gemm_fp8_blockwise: negative size");
    return MX_ERR_INVALID_ARG;
  }
  if (K % 128 != 0) {
    set_error("mx_gemm_fp8_blockwise: K must be a multiple of 128");
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  if (M > 0x7FFFFFFFLL || N > 0x7FFFFFFFLL || K > 0x7FFFFFFFLL) {
    set_error("mx_gemm_fp8_blockwise: sizes must be < 2^31");
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  mx_status st = check_output(c, ldc, N, M);
  if (st != MX_OK) return st;
  if (M == 0 || N == 0) return MX_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K > 0 && (!a_data || !b_data || !a_scale || !b_scale)) {
    set_error("mx_gemm_fp8_blockwise: null operand");
    return MX_ERR_INVALID_ARG;
  }
  if (K > 0 && (!aligned16(a_data) || !aligned16(b_data) || (reinterpret_cast<uintptr_t>(a_scale) & 3u) != 0 ||
                (reinterpret_cast<uintptr_t>(b_scale) & 3u) != 0)) {
    set_error("mx_gemm_fp8_blockwise: data must be 16-byte aligned, scales 4-byte aligned");
    return MX_ERR_ALIGNMENT;
  }
  st = check_device();
  if (st != MX_OK) return st;
  if (K == 0) return zero_output(c, ldc, N, M, s);
  GemmLaunch L;
  L.kind = GEMM_DENSE;
  L.a_data = a_data;
  L.a_scale = nullptr;
  L.a_ld = K;
  L.b_data = b_data;
  L.b_scale = nullptr;
  L.b_ld = K;
  L.M = M;
  L.N = N;
  L.K = K;
  L.b_rows_total = N;
  L.c = c;
  L.ldc = ldc;
  L.offsets = nullptr;
  L.n_groups = 0;
  L.dev_status = dev_status;
  L.bw_a_scale = a_scale;
  L.bw_b_scale = b_scale;
  return launch_gemm(L, s);
}

// Host checks and launch description of the rows-ragged gate_up fprop with
// the SwiGLU epilogue (shared by both SwiGLU entry points). *F is the number
// of output features (half of b's rows).
static mx_status swiglu_setup(const char* fn, const mx_operand* a, const mx_operand* b, const int64_t* group_offsets,
                              int n_groups, int* dev_status, GemmLaunch* L, int64_t* F) {
  mx_status st = check_operand(a, "a");
  if (st != MX_OK) return st;
  st = check_operand(b, "b");
  if (st != MX_OK) return st;
  st = check_mode(MX_FPROP, a, b);
  if (st != MX_OK) return st;
  if (!group_offsets || n_groups < 1) {
    set_error("%s: group_offsets must be non-null and n_groups >= 1", fn);
    return MX_ERR_INVALID_ARG;
  }
  if (n_groups > MX_MAX_GROUPS) {
    set_error("%s: n_groups = %d is above MX_MAX_GROUPS (%d)", fn, n_groups, MX_MAX_GROUPS);
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  if (a->k != b->k) {
    set_error("%s: a.k != b.k", fn);
    return MX_ERR_INVALID_ARG;
  }
  if (a->rows > 0x7FFFFFFFLL || b->rows > 0x7FFFFFFFLL || a->k > 0x7FFFFFFFLL) {
    set_error("%s: sizes must be < 2^31", fn);
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  if (b->rows % 256 != 0) {
    set_error("%s: gate_up rows (2F) must be a multiple of 256", fn);
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  *F = b->rows / 2;
  L->kind = GEMM_GROUPED_M;
  L->a_data = a->data;
  L->a_scale = a->scale;
  L->a_ld = a->ld ? a->ld : a->k;
  L->b_data = b->data;
  L->b_scale = b->scale;
  L->b_ld = b->ld ? b->ld : b->k;
  L->M = a->rows;
  L->N = b->rows;
  L->K = a->k;
  L->b_rows_total = b->rows * static_cast<int64_t>(n_groups);
  L->offsets = group_offsets;
  L->n_groups = n_groups;
  L->dev_status = dev_status;
  L->swiglu = true;
  return MX_OK;
}

mx_status mx_grouped_gemm_swiglu(const mx_operand* a, const mx_operand* b, const int64_t* group_offsets,
                                 int n_groups, void* c, int64_t ldc, int* dev_status, void* stream) {
  GemmLaunch L;
  int64_t F = 0;
  mx_status st = swiglu_setup("mx_grouped_gemm_swiglu", a, b, group_offsets, n_groups, dev_status, &L, &F);
  if (st != MX_OK) return st;
  st = check_output(c, ldc, F, a->rows);
  if (st != MX_OK) return st;
  if (a->rows == 0 || F == 0) return MX_OK;
  st = check_device();
  if (st != MX_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (a->k == 0) return zero_output(c, ldc, F, a->rows, s);  // silu(0) * 0
  L.c = c;
  L.ldc = ldc;
  return launch_gemm(L, s);
}

mx_status mx_grouped_gemm_swiglu_quantize(const mx_operand* a, const mx_operand* b, const int64_t* group_offsets,
                                          int n_groups, void* row_data, void* row_scale, void* col_data,
                                          void* col_scale, int64_t col_capacity, int* dev_status, void* stream) {
  const char* fn = "mx_grouped_gemm_swiglu_quantize";
  GemmLaunch L;
  int64_t F = 0;
  mx_status st = swiglu_setup(fn, a, b, group_offsets, n_groups, dev_status, &L, &F);
  if (st != MX_OK) return st;
  if (!row_data || !row_scale || !col_data || !col_scale) {
    set_error("%s: the four outputs must be non-null", fn);
    return MX_ERR_INVALID_ARG;
  }
  if (!aligned16(row_data) || !aligned16(row_scale) || !aligned16(col_data) || !aligned16(col_scale)) {
    set_error("%s: outputs must be 16-byte aligned", fn);
    return MX_ERR_ALIGNMENT;
  }
  if (a->rows == 0 || F == 0) return MX_OK;
  if (col_capacity < 128 || col_capacity % 128 != 0) {
    set_error("%s: col_capacity must be a positive multiple of 128 (at least the sum of the 128-padded groups)", fn);
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  st = check_device();
  if (st != MX_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (a->k == 0) {
    // silu(0) * 0 = 0 everywhere: zero codes and zero scales in both copies
    const size_t sizes[4] = {static_cast<size_t>(a->rows) * F, mx_scale_bytes(a->rows, F),
                             static_cast<size_t>(F) * col_capacity, mx_scale_bytes(F, col_capacity)};
    void* bufs[4] = {row_data, row_scale, col_data, col_scale};
    for (int i = 0; i < 4; ++i) {
      if (sizes[i] == 0) continue;
      st = cuda_status(cudaMemsetAsync(bufs[i], 0, sizes[i], s), "cudaMemsetAsync");
      if (st != MX_OK) return st;
    }
    return MX_OK;
  }
  L.q_row_data = row_data;
  L.q_row_scale = row_scale;
  L.q_col_data = col_data;
  L.q_col_scale = col_scale;
  L.q_cap = col_capacity;
  return launch_gemm(L, s);
}

mx_status mx_grouped_gemm(int mode, const mx_operand* a, const mx_operand* b, const int64_t* group_offsets,
                          int n_groups, void* c, int64_t ldc, int* dev_status, void* stream) {
  mx_status st = check_operand(a, "a");
  if (st != MX_OK) return st;
  st = check_operand(b, "b");
  if (st != MX_OK) return st;
  st = check_mode(mode, a, b);
  if (st != MX_OK) return st;
  if (!group_offsets || n_groups < 1) {
    set_error("mx_grouped_gemm: group_offsets must be non-null and n_groups >= 1");
    return MX_ERR_INVALID_ARG;
  }
  if (n_groups > MX_MAX_GROUPS) {
    set_error("mx_grouped_gemm: n_groups = %d is above MX_MAX_GROUPS (%d)", n_groups, MX_MAX_GROUPS);
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  if (a->k != b->k) {
    set_error("mx_grouped_gemm: a.k != b.k");
    return MX_ERR_INVALID_ARG;
  }
  if (a->rows > 0x7FFFFFFFLL || b->rows > 0x7FFFFFFFLL || a->k > 0x7FFFFFFFLL) {
    set_error("mx_grouped_gemm: sizes must be < 2^31");
    return MX_ERR_UNSUPPORTED_SHAPE;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  GemmLaunch L;
  L.a_data = a->data;
  L.a_scale = a->scale;
  L.a_ld = a->ld ? a->ld : a->k;
  L.b_data = b->data;
  L.b_scale = b->scale;
  L.b_ld = b->ld ? b->ld : b->k;
  L.K = a->k;
  L.c = c;
  L.ldc = ldc;
  L.offsets = group_offsets;
  L.n_groups = n_groups;
  L.dev_status = dev_status;
  if (mode == MX_WGRAD) {
    // c = [E, N, Kout]: N = a.rows (dY columns), Kout = b.rows (X columns).
    if (a->k % 128 != 0) {
      set_error("mx_grouped_gemm: wgrad capacity (a.k) must be a multiple of 128");
      return MX_ERR_UNSUPPORTED_SHAPE;
    }
    st = check_output(c, ldc, b->rows, a->rows * static_cast<int64_t>(n_groups));
    if (st != MX_OK) return st;
    if (a->rows == 0 || b->rows == 0) return MX_OK;
    st = check_device();
    if (st != MX_OK) return st;
    if (a->k == 0) return zero_output(c, ldc, b->rows, a->rows * static_cast<int64_t>(n_groups), s);
    L.kind = GEMM_GROUPED_K;
    L.M = a->rows;
    L.N = b->rows;
    L.b_rows_total = b->rows;
  } else {
    // a = [M_total, K] tokens grouped by expert; b = [E][N][K] stacked weights.
    st = check_output(c, ldc, b->rows, a->rows);
    if (st != MX_OK) return st;
    if (a->rows == 0 || b->rows == 0) return MX_OK;
    st = check_device();
    if (st != MX_OK) return st;
    if (a->k == 0) return zero_output(c, ldc, b->rows, a->rows, s);
    L.kind = GEMM_GROUPED_M;
    L.M = a->rows;
    L.N = b->rows;
    L.b_rows_total = b->rows * static_cast<int64_t>(n_groups);
  }
  return launch_gemm(L, s);
}

}  // extern "C"
