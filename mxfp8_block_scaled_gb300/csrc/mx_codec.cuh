// MX block codec shared by the quantiser and the GEMM epilogue that quantises
// its own output: the E8M0 scale rule, the E4M3 element conversion and the
// swizzled scale-atom layout ("浮点格式、数值稳定性与混合精度" §二.2, §三;
// "DeepSeek-V3 16B FSDP2 MXFP8/HiF8 训练设计" §3.1: 1x32 blocks, E8M0 scales).
//
// Scale rule: X = floor(log2 amax) - 8 clamped to [-127, 127], code X + 127;
// a block holding Inf or NaN gets code 0xFF. Elements: E4M3(x * 2^-X), round
// to nearest even, saturating at 448 (NaN blocks are handled by the callers).
#pragma once

#include <cuda_fp8.h>
#include <cstdint>

namespace mx {

// Byte offset of logical scale (r, kb) in the swizzled layout with `ka`
// scale-column atoms per 128-row band.
__device__ __forceinline__ int64_t scale_offset(int64_t r, int64_t kb, int64_t ka) {
  return (((r >> 7) * ka + (kb >> 2)) << 9) + ((r & 31) << 4) + (((r >> 5) & 3) << 2) + (kb & 3);
}

// E8M0 code from the largest BF16 magnitude pattern of a block.
__device__ __forceinline__ uint32_t scale_code(uint32_t amax_bits) {
  const int e = static_cast<int>(amax_bits >> 7);  // biased exponent, shared with FP32
  if (e == 0xFF) return 0xFFu;                     // block holds Inf or NaN
  const int x = e - 127 - 8;                       // floor(log2 amax) - 8 for normal amax
  return static_cast<uint32_t>(max(x, -127) + 127);
}

// 2**-X as an FP32 number (exponent field 254 - code, always normal).
__device__ __forceinline__ float inv_scale(uint32_t code) { return __uint_as_float((254u - code) << 23); }

__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two values -> two E4M3 bytes (a in the low byte).
__device__ __forceinline__ uint32_t cvt_pair(float a, float b) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

// NaN codes keeping the sign of the two BF16 halves of w.
__device__ __forceinline__ uint32_t nan_pair(uint32_t w) {
  return (0x7Fu | ((w >> 8) & 0x80u)) | ((0x7Fu | ((w >> 24) & 0x80u)) << 8);
}

// Quantise the two BF16 values of one word (low half -> low byte).
__device__ __forceinline__ uint32_t quant_word(uint32_t w, float inv) { return cvt_pair(lo_f(w) * inv, hi_f(w) * inv); }

// Four BF16 values (two words) -> four E4M3 bytes.
__device__ __forceinline__ uint32_t quant_quad(uint32_t a, uint32_t b, float inv) {
  return quant_word(a, inv) | (quant_word(b, inv) << 16);
}

__device__ __forceinline__ uint32_t half_max(uint32_t m) { return max(m & 0xFFFFu, m >> 16); }

}  // namespace mx
