// Device helpers of the NVFP4 format shared by the quantize kernels and the NVFP4 GEMM.
//
// Page: "Generalized Tensor Parallelism (GTP)" (Megatron-Core developer guide), §1.3 and
// "GTP + NVFP4": packed 4-bit E2M1 elements, one scale per 16 elements (table
// "Communication volume breakdown": 0.5 + 1/16 bytes per element), and a per-tensor scale
// set when the optimizer step quantizes.  The scale rule (two levels, every step in fp32):
//   S    = 1 if amax == 0, else min(2688 / amax, FLT_MAX)            2688 = 448 * 6
//   sf_b = RNE_E4M3_satfinite((amax_b / 6) * S)            one byte per block of 16
//   code = RNE_E2M1_satfinite(x * min(S / sf_b, FLT_MAX)), x * 0 when sf_b == 0
//   x   ~= e2m1(code) * sf_b / S
#pragma once

#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include <cfloat>
#include <cstdint>

namespace gtp {
namespace nv {

constexpr uint32_t kNanScale = 0x7Fu;  // E4M3 NaN: a block that holds NaN or Inf

__device__ __forceinline__ float tensor_scale(float amax) {
  if (amax == 0.f) return 1.f;
  return fminf(2688.f / amax, FLT_MAX);
}

__device__ __forceinline__ uint32_t block_scale_byte(float amax_b, float S) {
  const float d = (amax_b / 6.f) * S;
  return uint32_t(__nv_cvt_float_to_fp8(d, __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ float e4m3_value(uint32_t byte) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw(__nv_fp8_storage_t(byte), __NV_E4M3);
  return __half2float(__half(h));
}

// The element multiplier of a block: S / sf clamped to FLT_MAX (a clamped S over a tiny
// sf overflows), or 0 for a zero scale.
__device__ __forceinline__ float element_scale(uint32_t sbyte, float S) {
  const float sf = e4m3_value(sbyte);
  return sf == 0.f ? 0.f : fminf(S / sf, FLT_MAX);
}

// Two E2M1 codes of two already scaled values in one byte, the first in the low nibble.
__device__ __forceinline__ uint32_t encode2(float a, float b) {
  return uint32_t(__nv_cvt_float2_to_fp4x2(make_float2(a, b), __NV_E2M1, cudaRoundNearest));
}

}  // namespace nv
}  // namespace gtp
