// Device helpers of the MX block format shared by the quantize kernels and the optimizer
// sweep that writes MXFP8 weights directly.
//
// Page: "Generalized Tensor Parallelism (GTP)" (Megatron-Core developer guide), §1.3 and
// table "Communication volume breakdown": blocks of 32 elements, one scale byte each.
// Scale rule (OCP MX): E8M0 scale 2^(floor(log2 amax) - 8), 8 being the exponent of
// E4M3's largest power of two, clamped to the E8M0 range; each element is x / scale
// rounded to nearest-even E4M3 with saturation at +-448.  A block holding NaN or Inf gets
// scale byte 0xFF and elements 0x7F.
#pragma once

#include <cuda_fp8.h>

#include <cstdint>

namespace gtp {
namespace mx {

constexpr uint32_t kNanScale = 0xFFu;
constexpr uint32_t kNanCodes = 0x7F7F7F7Fu;  // four E4M3 NaN codes

// Scale byte of a block whose amax is finite.  floor(log2 amax) is the biased exponent
// minus 127 for a normal amax; zero and fp32 subnormals clamp to 2^-127 (byte 0), so
// byte = max(biased - 8, 0).  The largest finite amax gives byte 246.
__device__ __forceinline__ uint32_t scale_byte(float amax) {
  const int biased = int((__float_as_uint(amax) >> 23) & 0xFFu);
  return uint32_t(max(biased - 8, 0));
}

// 1 / scale = 2^(127 - byte): a normal float with biased exponent 254 - byte, so that
// x * inv_scale is an exact power-of-two scaling of x (up to fp32 underflow of values that
// round to zero in E4M3 anyway).
__device__ __forceinline__ float inv_scale(uint32_t sbyte) { return __uint_as_float((254u - sbyte) << 23); }

// Four E4M3 codes (little-endian in a word) of four already scaled values.
__device__ __forceinline__ uint32_t encode4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

}  // namespace mx
}  // namespace gtp
