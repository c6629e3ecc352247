// NVFP4 quantization of a weight (or activation) matrix: packed E2M1 elements, one E4M3
// scale byte per 16 consecutive elements of a row, and the tensor's amax from which the
// per-tensor scale follows.
//
// Page: "Generalized Tensor Parallelism (GTP)" (Megatron-Core developer guide), §1.3 and
// "GTP + NVFP4" (native NVFP4 parameters, packed 4-bit kFloat4E2M1, written by the
// optimizer once per step with the per-tensor scale set at that quantize; block 16 and
// 1/16 byte of scale per element in the table "Communication volume breakdown").  The
// scale rule is the one in nv_block.cuh.
//
// Two launches: a max-reduction of |x| over the finite elements into the caller's fp32
// amax (non-negative floats order like their bit patterns, so an integer atomicMax per
// block combines the block maxima), then the quantize pass: each thread owns 8
// consecutive elements, two neighbouring lanes one block of 16 (one shuffle combines the
// block's amax and its finite flag).  Purely HBM-bound: the source is read twice (4 or 2
// bytes per element each time), 0.5 + 1/16 bytes per element are written.
#include <cuda_bf16.h>

#include <algorithm>

#include "device.h"
#include "nv_block.cuh"
#include "sm100_ptx.cuh"

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void load8(const float *src, int64_t v, float (&x)[8]) {
  const float4 a = __ldcs(reinterpret_cast<const float4 *>(src) + 2 * v);
  const float4 b = __ldcs(reinterpret_cast<const float4 *>(src) + 2 * v + 1);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

__device__ __forceinline__ void load8(const __nv_bfloat16 *src, int64_t v, float (&x)[8]) {
  const uint4 a = __ldcs(reinterpret_cast<const uint4 *>(src) + v);
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);  // bf16 -> fp32 is exact
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) nv_amax_kernel(const T *__restrict__ src, int64_t nvec,
                                                           unsigned int *__restrict__ amax_bits) {
  __shared__ float red[kThreads / 32];
  gtp::ptx::allow_dependents();
  gtp::ptx::wait_prior_grid();
  float m = 0.f;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t v = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; v < nvec; v += stride) {
    float x[8];
    load8(src, v, x);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (isfinite(x[i])) m = fmaxf(m, fabsf(x[i]));
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, d));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = red[0];
    for (int w = 1; w < kThreads / 32; ++w) b = fmaxf(b, red[w]);
    atomicMax(amax_bits, __float_as_uint(b));
  }
}

// Scale byte (row r, column j) of a [rows, C] scale array: at r * C + j, or at its place
// in the tiled layout (gtp_sf_tile) when `words` (= ceil(C / 4)) is non-zero.
__device__ __forceinline__ int64_t scale_index(int64_t b, int64_t C, int64_t words) {
  if (words == 0) return b;
  const int64_t r = b / C, j = b - r * C;
  return ((r >> 7) * words + (j >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (j & 3);
}

template <typename T>
__global__ void __launch_bounds__(kThreads) nv_quantize_kernel(const T *__restrict__ src, int64_t nvec,
                                                               const float *__restrict__ amax,
                                                               uint8_t *__restrict__ packed,
                                                               uint8_t *__restrict__ scale, int64_t C,
                                                               int64_t words) {
  gtp::ptx::allow_dependents();
  gtp::ptx::wait_prior_grid();
  const float S = gtp::nv::tensor_scale(__ldg(amax));
  const int lane = threadIdx.x & 31;
  const unsigned pair = 0x3u << (lane & ~1);  // the 2 lanes that share a 16-element block
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t v = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; v < nvec; v += stride) {
    float x[8];
    load8(src, v, x);
    float amax_b = 0.f;
    bool finite = true;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      finite = finite && isfinite(x[i]);
      amax_b = fmaxf(amax_b, fabsf(x[i]));
    }
    amax_b = fmaxf(amax_b, __shfl_xor_sync(pair, amax_b, 1));
    const int fin = (finite ? 1 : 0) & __shfl_xor_sync(pair, finite ? 1 : 0, 1);
    uint32_t sbyte, word = 0;
    if (fin) {
      sbyte = gtp::nv::block_scale_byte(amax_b, S);
      const float e = gtp::nv::element_scale(sbyte, S);
#pragma unroll
      for (int i = 0; i < 4; ++i) word |= gtp::nv::encode2(x[2 * i] * e, x[2 * i + 1] * e) << (8 * i);
    } else {
      sbyte = gtp::nv::kNanScale;
    }
    __stcs(reinterpret_cast<uint32_t *>(packed) + v, word);
    if ((lane & 1) == 0) scale[scale_index(v >> 1, C, words)] = uint8_t(sbyte);
  }
}

}  // namespace

namespace {

gtp_status quantize(const void *src, gtp_dtype src_dt, int64_t rows, int64_t cols, uint8_t *packed, uint8_t *scales,
                    float *amax, bool tiled, gtp_stream stream) {
  gtp::clear_error();
  if (src_dt != GTP_F32 && src_dt != GTP_BF16) return gtp::fail(GTP_E_DTYPE, "src must be F32 or BF16");
  if (rows < 0 || cols < 0) return gtp::fail(GTP_E_ARG, "negative size");
  if (cols % 16) return gtp::fail(GTP_E_SHAPE, "cols must be a multiple of 16");
  if (rows > (int64_t(1) << 40) / (cols ? cols : 1)) return gtp::fail(GTP_E_SHAPE, "matrix too large");
  if (!amax) return gtp::fail(GTP_E_ARG, "null amax");
  if (reinterpret_cast<uintptr_t>(amax) & 3u) return gtp::fail(GTP_E_ALIGN, "amax must be 4-byte aligned");
  if (rows > 0 && cols > 0) {
    if (!src || !packed || !scales) return gtp::fail(GTP_E_ARG, "null pointer");
    if (!gtp::aligned16(src) || !gtp::aligned16(packed))
      return gtp::fail(GTP_E_ALIGN, "src and packed must be 16-byte aligned");
  }
  gtp::DeviceInfo dev;
  if (gtp_status s = gtp::require_sm103(&dev)) return s;
  cudaStream_t st = gtp::as_stream(stream);
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), st);
  if (e != cudaSuccess) return gtp::fail(GTP_E_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));
  if (rows == 0 || cols == 0) return GTP_OK;  // amax 0: the tensor scale is 1
  const int64_t nvec = rows * cols / 8;
  const int64_t C = cols / 16, words = tiled ? (C + 3) / 4 : 0;
  const int64_t want = (nvec + kThreads - 1) / kThreads;
  const int grid = int(std::max<int64_t>(1, std::min<int64_t>(want, int64_t(dev.sm_count) * 8)));
  auto *bits = reinterpret_cast<unsigned int *>(amax);
  if (src_dt == GTP_F32) {
    auto *s = static_cast<const float *>(src);
    if (gtp_status r = gtp::launch_overlapped(nv_amax_kernel<float>, grid, kThreads, 0, st, "nvfp4_amax", s, nvec,
                                              bits))
      return r;
    return gtp::launch_overlapped(nv_quantize_kernel<float>, grid, kThreads, 0, st, "nvfp4_quantize_rowwise", s, nvec,
                                  const_cast<const float *>(amax), packed, scales, C, words);
  }
  auto *s = static_cast<const __nv_bfloat16 *>(src);
  if (gtp_status r = gtp::launch_overlapped(nv_amax_kernel<__nv_bfloat16>, grid, kThreads, 0, st, "nvfp4_amax", s,
                                            nvec, bits))
    return r;
  return gtp::launch_overlapped(nv_quantize_kernel<__nv_bfloat16>, grid, kThreads, 0, st, "nvfp4_quantize_rowwise", s,
                                nvec, const_cast<const float *>(amax), packed, scales, C, words);
}

}  // namespace

extern "C" gtp_status gtp_nvfp4_quantize_rowwise(const void *src, gtp_dtype src_dt, int64_t rows, int64_t cols,
                                                 uint8_t *packed, uint8_t *scales, float *amax, gtp_stream stream) {
  return quantize(src, src_dt, rows, cols, packed, scales, amax, false, stream);
}

extern "C" gtp_status gtp_nvfp4_quantize_rowwise_tiled(const void *src, gtp_dtype src_dt, int64_t rows, int64_t cols,
                                                       uint8_t *packed, uint8_t *scales_tiled, float *amax,
                                                       gtp_stream stream) {
  return quantize(src, src_dt, rows, cols, packed, scales_tiled, amax, true, stream);
}
