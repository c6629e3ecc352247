// MX block quantization of a weight (or activation) matrix: E4M3 elements plus one E8M0
// scale byte per 32 consecutive elements of a row.
//
// Page: "Generalized Tensor Parallelism (GTP)" (Megatron-Core developer guide), §1.3: native
// MXFP8 weights, block 32 with 1/32 byte of scale per element, written from the fp32
// master once per optimizer step.  The scale rule is the OCP MX one: the scale of a
// block is 2^(floor(log2 amax) - 8) (8 = exponent of E4M3's largest power of two),
// clamped to the E8M0 range, and each element is rounded to nearest-even E4M3 after
// division by it, saturating at +-448.  A block that holds NaN or Inf gets scale 0xFF
// and elements 0x7F.
//
// Layout of the work: each thread owns 8 consecutive elements (32 bytes of fp32 or 16 of
// bf16), four neighbouring lanes own one block; the block's amax and "has a non-finite
// value" flag are combined with two butterfly shuffles inside the 4-lane group.  Purely
// HBM-bound: read 4 (or 2) bytes, write 1 + 1/32 bytes per element.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "device.h"
#include "mx_block.cuh"
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
    x[2 * i] = __uint_as_float(w[i] << 16);              // bf16 -> fp32 is exact
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
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
__global__ void __launch_bounds__(kThreads) mx_quantize_kernel(const T *__restrict__ src, int64_t nvec,
                                                               uint8_t *__restrict__ q, uint8_t *__restrict__ scale,
                                                               int64_t C, int64_t words) {
  gtp::ptx::allow_dependents();
  gtp::ptx::wait_prior_grid();
  const int lane = threadIdx.x & 31;
  const unsigned group = 0xFu << (lane & ~3);   // the 4 lanes that share a 32-element block
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t v = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; v < nvec; v += stride) {
    float x[8];
    load8(src, v, x);
    float amax = 0.f;
    bool finite = true;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      finite = finite && isfinite(x[i]);
      amax = fmaxf(amax, fabsf(x[i]));
    }
    amax = fmaxf(amax, __shfl_xor_sync(group, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(group, amax, 2));
    int fin = finite ? 1 : 0;
    fin &= __shfl_xor_sync(group, fin, 1);
    fin &= __shfl_xor_sync(group, fin, 2);
    uint32_t sbyte;
    uint2 packed;
    if (fin) {
      sbyte = gtp::mx::scale_byte(amax);
      const float inv = gtp::mx::inv_scale(sbyte);
      packed.x = gtp::mx::encode4(x[0] * inv, x[1] * inv, x[2] * inv, x[3] * inv);
      packed.y = gtp::mx::encode4(x[4] * inv, x[5] * inv, x[6] * inv, x[7] * inv);
    } else {
      sbyte = gtp::mx::kNanScale;
      packed = make_uint2(gtp::mx::kNanCodes, gtp::mx::kNanCodes);
    }
    __stcs(reinterpret_cast<uint2 *>(q) + v, packed);
    if ((lane & 3) == 0) scale[scale_index(v >> 2, C, words)] = uint8_t(sbyte);
  }
}

// Columnwise (backward) view: blocks of 32 consecutive rows of one column, written
// transposed, so that the column's 32-blocks are contiguous in a row of the output
// (q_t[c][r], s_t[c][r / 32]).  A thread owns V adjacent columns (2 when the row length
// and the source alignment allow one 2-element load, else 1) of kColStrips 32-row strips,
// taken one after the other: per strip it reads the 32 rows of its columns (each read is
// coalesced across the block), reduces each column's amax in registers and writes 32
// contiguous E4M3 bytes per column; the strips' scale bytes of a column go out as one
// 2-byte store where the scale rows allow it.  Measured on the MXFP8 workload's three
// sources: 2 columns x 2 strips in 64-thread blocks ran 12 % faster than 1 x 1 in
// 128-thread blocks; 4 columns, 4 strips or 256-thread blocks were slower.
constexpr int kColThreads = 64;
constexpr int kColStrips = 2;  // 32-row strips a thread takes, one after the other

// V adjacent elements of one row, as one load.
template <typename T, int V>
__device__ __forceinline__ void loadv(const T *src, int64_t i, float (&x)[V]);
template <>
__device__ __forceinline__ void loadv<float, 1>(const float *src, int64_t i, float (&x)[1]) { x[0] = __ldcs(src + i); }
template <>
__device__ __forceinline__ void loadv<float, 2>(const float *src, int64_t i, float (&x)[2]) {
  const float2 a = __ldcs(reinterpret_cast<const float2 *>(src + i));
  x[0] = a.x;
  x[1] = a.y;
}
template <>
__device__ __forceinline__ void loadv<__nv_bfloat16, 1>(const __nv_bfloat16 *src, int64_t i, float (&x)[1]) {
  x[0] = __uint_as_float(uint32_t(__ldcs(reinterpret_cast<const unsigned short *>(src) + i)) << 16);
}
template <>
__device__ __forceinline__ void loadv<__nv_bfloat16, 2>(const __nv_bfloat16 *src, int64_t i, float (&x)[2]) {
  const uint32_t w = __ldcs(reinterpret_cast<const unsigned int *>(src + i));
  x[0] = __uint_as_float(w << 16);
  x[1] = __uint_as_float(w & 0xFFFF0000u);
}

template <typename T, int V, int S>
__global__ void __launch_bounds__(kColThreads) mx_quantize_col_kernel(const T *__restrict__ src, int64_t rows,
                                                                      int64_t cols, uint8_t *__restrict__ qt,
                                                                      uint8_t *__restrict__ st, int pack) {
  gtp::ptx::allow_dependents();
  gtp::ptx::wait_prior_grid();
  const int64_t c = (int64_t(blockIdx.x) * kColThreads + threadIdx.x) * V;
  if (c >= cols) return;
  const int64_t strips = rows / 32;
  const int64_t s0 = int64_t(blockIdx.y) * S;
  uint32_t sc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) sc[v] = 0;
#pragma unroll
  for (int s = 0; s < S; ++s) {
    if (s0 + s >= strips) break;
    const int64_t r0 = (s0 + s) * 32;
    float x[V][32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      float t[V];
      loadv<T, V>(src, (r0 + i) * cols + c, t);
#pragma unroll
      for (int v = 0; v < V; ++v) x[v][i] = t[v];
    }
#pragma unroll
    for (int v = 0; v < V; ++v) {
      float amax = 0.f;
      bool finite = true;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        finite = finite && isfinite(x[v][i]);
        amax = fmaxf(amax, fabsf(x[v][i]));
      }
      uint32_t w[8];
      uint32_t sbyte;
      if (finite) {
        sbyte = gtp::mx::scale_byte(amax);
        const float inv = gtp::mx::inv_scale(sbyte);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          w[i] = gtp::mx::encode4(x[v][4 * i] * inv, x[v][4 * i + 1] * inv, x[v][4 * i + 2] * inv,
                                  x[v][4 * i + 3] * inv);
      } else {
        sbyte = gtp::mx::kNanScale;
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = gtp::mx::kNanCodes;
      }
      uint4 *dst = reinterpret_cast<uint4 *>(qt + (c + v) * rows + r0);
      __stcs(dst, make_uint4(w[0], w[1], w[2], w[3]));
      __stcs(dst + 1, make_uint4(w[4], w[5], w[6], w[7]));
      if (S == 1) st[(c + v) * strips + s0] = uint8_t(sbyte);
      else sc[v] |= sbyte << (8 * s);
    }
  }
  if (S > 1) {
    const int ns = int(strips - s0 < S ? strips - s0 : S);
#pragma unroll
    for (int v = 0; v < V; ++v) {
      uint8_t *p = st + (c + v) * strips + s0;
      if (pack && ns == S) {
        if (S == 4) *reinterpret_cast<uint32_t *>(p) = sc[v];
        else *reinterpret_cast<uint16_t *>(p) = uint16_t(sc[v]);
      } else {
        for (int s = 0; s < ns; ++s) p[s] = uint8_t(sc[v] >> (8 * s));
      }
    }
  }
}

template <typename T, int V>
gtp_status launch_col_v(const T *src, int64_t rows, int64_t cols, uint8_t *qt, uint8_t *st, cudaStream_t stream) {
  const int64_t strips = rows / 32;
  const int64_t gy = (strips + kColStrips - 1) / kColStrips;
  if (gy > 65535) return gtp::fail(GTP_E_SHAPE, "rows / %d above 65535", 32 * kColStrips);
  const dim3 grid{unsigned((cols / V + kColThreads - 1) / kColThreads), unsigned(gy)};
  const int pack = (strips % kColStrips == 0 && reinterpret_cast<uintptr_t>(st) % kColStrips == 0) ? 1 : 0;
  return gtp::launch_overlapped(mx_quantize_col_kernel<T, V, kColStrips>, grid, kColThreads, 0, stream,
                                "mxfp8_quantize_columnwise", src, rows, cols, qt, st, pack);
}

template <typename T>
gtp_status launch_col(const T *src, int64_t rows, int64_t cols, uint8_t *qt, uint8_t *st, cudaStream_t stream) {
  if (cols % 2 == 0 && reinterpret_cast<uintptr_t>(src) % (2 * sizeof(T)) == 0)
    return launch_col_v<T, 2>(src, rows, cols, qt, st, stream);
  return launch_col_v<T, 1>(src, rows, cols, qt, st, stream);
}

}  // namespace

extern "C" gtp_status gtp_mxfp8_quantize_columnwise(const void *src, gtp_dtype src_dt, int64_t rows, int64_t cols,
                                                    uint8_t *e4m3_t, uint8_t *e8m0_t, gtp_stream stream) {
  gtp::clear_error();
  if (src_dt != GTP_F32 && src_dt != GTP_BF16) return gtp::fail(GTP_E_DTYPE, "src must be F32 or BF16");
  if (rows < 0 || cols < 0) return gtp::fail(GTP_E_ARG, "negative size");
  if (rows % 32) return gtp::fail(GTP_E_SHAPE, "rows must be a multiple of 32");
  if (cols > (int64_t(1) << 31) || rows > (int64_t(1) << 36) / (cols ? cols : 1))
    return gtp::fail(GTP_E_SHAPE, "matrix too large");
  if (rows == 0 || cols == 0) return GTP_OK;
  if (!src || !e4m3_t || !e8m0_t) return gtp::fail(GTP_E_ARG, "null pointer");
  if (!gtp::aligned16(e4m3_t)) return gtp::fail(GTP_E_ALIGN, "e4m3_t must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(src) & (src_dt == GTP_F32 ? 3u : 1u)) return gtp::fail(GTP_E_ALIGN, "src alignment");
  if (rows / 32 > 65535) return gtp::fail(GTP_E_SHAPE, "rows / 32 above 65535");
  gtp::DeviceInfo dev;
  if (gtp_status s = gtp::require_sm103(&dev)) return s;
  cudaStream_t st = gtp::as_stream(stream);
  if (src_dt == GTP_F32) return launch_col(static_cast<const float *>(src), rows, cols, e4m3_t, e8m0_t, st);
  return launch_col(static_cast<const __nv_bfloat16 *>(src), rows, cols, e4m3_t, e8m0_t, st);
}

namespace {

gtp_status quantize_rowwise(const void *src, gtp_dtype src_dt, int64_t rows, int64_t cols, uint8_t *e4m3,
                            uint8_t *e8m0, bool tiled, gtp_stream stream) {
  gtp::clear_error();
  if (src_dt != GTP_F32 && src_dt != GTP_BF16) return gtp::fail(GTP_E_DTYPE, "src must be F32 or BF16");
  if (rows < 0 || cols < 0) return gtp::fail(GTP_E_ARG, "negative size");
  if (cols % 32) return gtp::fail(GTP_E_SHAPE, "cols must be a multiple of 32");
  if (rows > (int64_t(1) << 40) / (cols ? cols : 1)) return gtp::fail(GTP_E_SHAPE, "matrix too large");
  if (rows == 0 || cols == 0) return GTP_OK;
  if (!src || !e4m3 || !e8m0) return gtp::fail(GTP_E_ARG, "null pointer");
  if (!gtp::aligned16(src) || !gtp::aligned16(e4m3)) return gtp::fail(GTP_E_ALIGN, "src and e4m3 must be 16-byte aligned");
  gtp::DeviceInfo dev;
  if (gtp_status s = gtp::require_sm103(&dev)) return s;
  const int64_t nvec = rows * cols / 8;
  const int64_t C = cols / 32, words = tiled ? (C + 3) / 4 : 0;
  const int64_t want = (nvec + kThreads - 1) / kThreads;
  const int grid = int(std::max<int64_t>(1, std::min<int64_t>(want, int64_t(dev.sm_count) * 8)));
  cudaStream_t st = gtp::as_stream(stream);
  if (src_dt == GTP_F32)
    return gtp::launch_overlapped(mx_quantize_kernel<float>, grid, kThreads, 0, st, "mxfp8_quantize_rowwise",
                                  static_cast<const float *>(src), nvec, e4m3, e8m0, C, words);
  return gtp::launch_overlapped(mx_quantize_kernel<__nv_bfloat16>, grid, kThreads, 0, st, "mxfp8_quantize_rowwise",
                                static_cast<const __nv_bfloat16 *>(src), nvec, e4m3, e8m0, C, words);
}

}  // namespace

extern "C" gtp_status gtp_mxfp8_quantize_rowwise(const void *src, gtp_dtype src_dt, int64_t rows, int64_t cols,
                                                 uint8_t *e4m3, uint8_t *e8m0, gtp_stream stream) {
  return quantize_rowwise(src, src_dt, rows, cols, e4m3, e8m0, false, stream);
}

extern "C" gtp_status gtp_mxfp8_quantize_rowwise_tiled(const void *src, gtp_dtype src_dt, int64_t rows, int64_t cols,
                                                       uint8_t *e4m3, uint8_t *e8m0_tiled, gtp_stream stream) {
  return quantize_rowwise(src, src_dt, rows, cols, e4m3, e8m0_tiled, true, stream);
}
