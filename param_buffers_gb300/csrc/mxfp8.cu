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
// bf16), four neighbouring lanes own one block; the block's amax, kept as the largest |x|
// bit pattern (which also flags NaN and Inf), is combined with two butterfly shuffles
// inside the 4-lane group.  Purely
// HBM-bound: read 4 (or 2) bytes, write 1 + 1/32 bytes per element.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>

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

// The same for scale (r, j) of a [R, C] array given as its row and column.
__device__ __forceinline__ int64_t scale_index_rc(int64_t r, int64_t j, int64_t C, int64_t words) {
  if (words == 0) return r * C + j;
  return ((r >> 7) * words + (j >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (j & 3);
}

// Vector v (elements 8 v .. 8 v + 7) of a row-major matrix whose rows are C blocks long:
// its codes, and the block's scale byte from the first of the block's four lanes.  The
// four lanes of a block (lanes 4 k .. 4 k + 3) must take part together.
template <typename T>
__device__ __forceinline__ void row_vec(const T *__restrict__ src, int64_t v, uint8_t *__restrict__ q,
                                        uint8_t *__restrict__ scale, int64_t C, int64_t words, int lane) {
  const unsigned group = 0xFu << (lane & ~3);   // the 4 lanes that share a 32-element block
  float x[8];
  load8(src, v, x);
  // the block's largest |x| bit pattern: its amax, and at or above 0x7F800000 exactly when
  // the block holds NaN or Inf (they sort above every finite value)
  uint32_t abits = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) abits = max(abits, __float_as_uint(x[i]) & 0x7FFFFFFFu);
  abits = max(abits, __shfl_xor_sync(group, abits, 1));
  abits = max(abits, __shfl_xor_sync(group, abits, 2));
  uint32_t sbyte;
  uint2 packed;
  if (abits < 0x7F800000u) {
    sbyte = gtp::mx::scale_byte(__uint_as_float(abits));
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

template <typename T>
__global__ void __launch_bounds__(kThreads) mx_quantize_kernel(const T *__restrict__ src, int64_t nvec,
                                                               uint8_t *__restrict__ q, uint8_t *__restrict__ scale,
                                                               int64_t C, int64_t words) {
  gtp::ptx::allow_dependents();
  gtp::ptx::wait_prior_grid();
  const int lane = threadIdx.x & 31;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t v = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; v < nvec; v += stride)
    row_vec(src, v, q, scale, C, words, lane);
}

// Several matrices in one launch: the grid strides through each matrix's vectors in turn
// (a matrix's vector count is a multiple of 4, so a block's four lanes stay together).
constexpr int kRowItems = 8;
struct RowItem {
  const void *src;
  uint8_t *q, *scale;
  int64_t nvec, C, words;
  int32_t bf16;
  int32_t pad;
};
struct RowArgs {
  RowItem it[kRowItems];
  int32_t n;
};

__global__ void __launch_bounds__(kThreads) mx_quantize_group_kernel(const __grid_constant__ RowArgs a) {
  gtp::ptx::allow_dependents();
  gtp::ptx::wait_prior_grid();
  const int lane = threadIdx.x & 31;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const int64_t t0 = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  for (int i = 0; i < a.n; ++i) {
    const RowItem &it = a.it[i];
    if (it.bf16) {
      for (int64_t v = t0; v < it.nvec; v += stride)
        row_vec(static_cast<const __nv_bfloat16 *>(it.src), v, it.q, it.scale, it.C, it.words, lane);
    } else {
      for (int64_t v = t0; v < it.nvec; v += stride)
        row_vec(static_cast<const float *>(it.src), v, it.q, it.scale, it.C, it.words, lane);
    }
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
                                                                      uint8_t *__restrict__ st, int pack,
                                                                      int64_t words) {
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
      // the largest |x| bit pattern: the amax, and above 0x7F7FFFFF for NaN or Inf
      uint32_t abits = 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) abits = max(abits, __float_as_uint(x[v][i]) & 0x7FFFFFFFu);
      const bool finite = abits < 0x7F800000u;
      const float amax = __uint_as_float(abits);
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
      if (S == 1) st[scale_index_rc(c + v, s0, strips, words)] = uint8_t(sbyte);
      else sc[v] |= sbyte << (8 * s);
    }
  }
  if (S > 1) {
    const int ns = int(strips - s0 < S ? strips - s0 : S);
#pragma unroll
    for (int v = 0; v < V; ++v) {
      if (pack && ns == S) {  // the S bytes are adjacent in either layout (s0 a multiple of S)
        uint8_t *p = st + scale_index_rc(c + v, s0, strips, words);
        if (S == 4) *reinterpret_cast<uint32_t *>(p) = sc[v];
        else *reinterpret_cast<uint16_t *>(p) = uint16_t(sc[v]);
      } else {
        for (int s = 0; s < ns; ++s) st[scale_index_rc(c + v, s0 + s, strips, words)] = uint8_t(sc[v] >> (8 * s));
      }
    }
  }
}

// words: 0 for [cols, rows / 32] scales, else the tiled layout's words a row (rows / 128, rounded up)
template <typename T, int V>
gtp_status launch_col_v(const T *src, int64_t rows, int64_t cols, uint8_t *qt, uint8_t *st, int64_t words,
                        cudaStream_t stream) {
  const int64_t strips = rows / 32;
  const int64_t gy = (strips + kColStrips - 1) / kColStrips;
  if (gy > 65535) return gtp::fail(GTP_E_SHAPE, "rows / %d above 65535", 32 * kColStrips);
  const dim3 grid{unsigned((cols / V + kColThreads - 1) / kColThreads), unsigned(gy)};
  // tiled scales: a 16-byte aligned array whose strips s0, s0 + 1 (s0 even) are adjacent bytes
  const int pack = words ? 1
                         : (strips % kColStrips == 0 && reinterpret_cast<uintptr_t>(st) % kColStrips == 0) ? 1 : 0;
  return gtp::launch_overlapped(mx_quantize_col_kernel<T, V, kColStrips>, grid, kColThreads, 0, stream,
                                "mxfp8_quantize_columnwise", src, rows, cols, qt, st, pack, words);
}

// Columnwise, warp tiles.  A warp quantizes one 32-row strip of a column tile that is
// 8 x VE columns wide (VE = 16 bytes of source elements: 4 fp32 or 8 bf16): lane 8 g + q
// reads rows g, g + 4, ..., g + 28 of columns VE q .. VE q + VE - 1, one 16-byte load a
// row (each load instruction covers four whole 128-byte row segments).  A column's amax,
// kept as the largest |x| bit pattern (which also flags NaN and Inf), is finished by two
// shuffles across the four lanes that share q.  The lane then encodes its 8 rows x VE columns; rows of a column sit in
// four lanes, interleaved by g, so the four lanes trade encoded words (three shuffle
// rounds) until lane g holds rows 8 g .. 8 g + 7 of each of its columns, which it writes
// as one 8-byte store a column: the four lanes of a column fill its 32-byte run of the
// transposed output.  The warp takes S strips one after the other and packs each
// column's S scale bytes into one store where the scale rows allow.  The warps of a block
// take adjacent column tiles of the same strips.
template <typename T>
struct ColTile;
// Column amax as bit patterns: for a non-negative float the bit pattern orders as the
// value does, and NaN and Inf sit above every finite value, so the largest |x| pattern
// of a column both gives the amax and flags a non-finite block (>= 0x7F800000).
template <>
struct ColTile<float> {
  static constexpr int VE = 4;
  __device__ static float at(const uint4 &w, int j) { return __uint_as_float((&w.x)[j]); }
  // a[j]: the largest |x| bit pattern of column j over this lane's 8 rows
  __device__ static void amax_bits(const uint4 (&w)[8], uint32_t (&a)[4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      a[j] = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) a[j] = max(a[j], (&w[i].x)[j] & 0x7FFFFFFFu);
    }
  }
  __device__ static uint32_t combine(uint32_t x, uint32_t y) { return max(x, y); }
  __device__ static uint32_t col_bits(const uint32_t (&a)[4], int j) { return a[j]; }
};
template <>
struct ColTile<__nv_bfloat16> {
  static constexpr int VE = 8;
  __device__ static float at(const uint4 &w, int j) {  // bf16 -> fp32 is exact
    const uint32_t x = (&w.x)[j >> 1];
    return __uint_as_float((j & 1) ? (x & 0xFFFF0000u) : (x << 16));
  }
  __device__ static uint32_t max2(uint32_t x, uint32_t y) {  // per 16-bit half, unsigned
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(x), "r"(y));
    return d;
  }
  // a[k]: the largest |x| bf16 patterns of columns 2k (low half) and 2k + 1 (high half)
  __device__ static void amax_bits(const uint4 (&w)[8], uint32_t (&a)[4]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      a[k] = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) a[k] = max2(a[k], (&w[i].x)[k] & 0x7FFF7FFFu);
    }
  }
  __device__ static uint32_t combine(uint32_t x, uint32_t y) { return max2(x, y); }
  __device__ static uint32_t col_bits(const uint32_t (&a)[4], int j) {
    return (j & 1) ? (a[j >> 1] & 0xFFFF0000u) : (a[j >> 1] << 16);
  }
};

// Swaps the word pairs of a 4-entry table so that entry k holds what was at k ^ g.
__device__ __forceinline__ void xor_permute(uint32_t (&a)[4], uint32_t (&b)[4], int g) {
  if (g & 1) {
    uint32_t t;
    t = a[0]; a[0] = a[1]; a[1] = t; t = a[2]; a[2] = a[3]; a[3] = t;
    t = b[0]; b[0] = b[1]; b[1] = t; t = b[2]; b[2] = b[3]; b[3] = t;
  }
  if (g & 2) {
    uint32_t t;
    t = a[0]; a[0] = a[2]; a[2] = t; t = a[1]; a[1] = a[3]; a[3] = t;
    t = b[0]; b[0] = b[2]; b[2] = t; t = b[1]; b[1] = b[3]; b[3] = t;
  }
}

// 4 x 4 byte transpose: byte j of out[i] = byte i of in[j].
__device__ __forceinline__ void transpose4x4(const uint32_t (&in)[4], uint32_t (&out)[4]) {
  const uint32_t lo01 = __byte_perm(in[0], in[1], 0x5140), hi01 = __byte_perm(in[0], in[1], 0x7362);
  const uint32_t lo23 = __byte_perm(in[2], in[3], 0x5140), hi23 = __byte_perm(in[2], in[3], 0x7362);
  out[0] = __byte_perm(lo01, lo23, 0x5410);
  out[1] = __byte_perm(lo01, lo23, 0x7632);
  out[2] = __byte_perm(hi01, hi23, 0x5410);
  out[3] = __byte_perm(hi01, hi23, 0x7632);
}

// Two warps a block: small blocks spread the warp tiles evenly over the SMs (measured on
// the workload's sources: the three-view group 6.24 TB/s against 5.85 with eight warps).
constexpr int kColTileThreads = 64;

// One loaded warp tile (w: this lane's 8 rows g + 4 i of columns c .. c + VE - 1 of the
// strip at row r0): its codes stored to the transposed output, the scale byte of column
// 4 u + g returned in sb[u].
template <typename T>
__device__ __forceinline__ void col_unit(const uint4 (&w)[8], uint8_t *__restrict__ qt, int64_t rows, int64_t c,
                                         int64_t r0, bool live, int g, uint32_t (&sb)[ColTile<T>::VE / 4]) {
  constexpr int VE = ColTile<T>::VE, NQ = VE / 4;
  uint32_t am[4];
  ColTile<T>::amax_bits(w, am);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    am[k] = ColTile<T>::combine(am[k], __shfl_xor_sync(0xFFFFFFFFu, am[k], 8));
    am[k] = ColTile<T>::combine(am[k], __shfl_xor_sync(0xFFFFFFFFu, am[k], 16));
  }
  uint32_t bad = 0;  // bit j: column j holds NaN or Inf
  float inv[VE];
  uint32_t sbyte[VE];
#pragma unroll
  for (int j = 0; j < VE; ++j) {
    const uint32_t bits = ColTile<T>::col_bits(am, j);
    if (bits >= 0x7F800000u) bad |= 1u << j;
    sbyte[j] = bits >= 0x7F800000u ? gtp::mx::kNanScale : gtp::mx::scale_byte(__uint_as_float(bits));
    inv[j] = gtp::mx::inv_scale(bits >= 0x7F800000u ? 0u : sbyte[j]);
  }
#pragma unroll
  for (int u = 0; u < NQ; ++u) {
    // codes of columns 4u .. 4u + 3 (bytes 0-3) of row g + 4 i, in word e[i]
    uint32_t nan_bytes = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (bad >> (4 * u + j) & 1u) nan_bytes |= 0xFFu << (8 * j);
    uint32_t e[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t code = gtp::mx::encode4(
          ColTile<T>::at(w[i], 4 * u) * inv[4 * u], ColTile<T>::at(w[i], 4 * u + 1) * inv[4 * u + 1],
          ColTile<T>::at(w[i], 4 * u + 2) * inv[4 * u + 2], ColTile<T>::at(w[i], 4 * u + 3) * inv[4 * u + 3]);
      e[i] = (code & ~nan_bytes) | (gtp::mx::kNanCodes & nan_bytes);
    }
    // lane g owes lane h the words of rows 8 h .. 8 h + 7: e[2 h] (rows 8h + g) and
    // e[2 h + 1] (rows 8h + 4 + g).  Entry k of (a, b) goes to lane g ^ k.
    uint32_t a[4] = {e[0], e[2], e[4], e[6]}, b[4] = {e[1], e[3], e[5], e[7]};
    xor_permute(a, b, g);
#pragma unroll
    for (int k = 1; k < 4; ++k) {
      a[k] = __shfl_xor_sync(0xFFFFFFFFu, a[k], 8 * k);
      b[k] = __shfl_xor_sync(0xFFFFFFFFu, b[k], 8 * k);
    }
    xor_permute(a, b, g);  // entry k now came from lane k: rows 8 g + k (a) and 8 g + 4 + k (b)
    uint32_t lo[4], hi[4];
    transpose4x4(a, lo);  // lo[j]: column 4u + j, rows 8 g .. 8 g + 3
    transpose4x4(b, hi);  //                       rows 8 g + 4 .. 8 g + 7
    if (live) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        __stcs(reinterpret_cast<uint2 *>(qt + (c + 4 * u + j) * rows + r0 + 8 * g), make_uint2(lo[j], hi[j]));
    }
    uint32_t mine = sbyte[4 * u];  // lane g keeps the scale byte of column 4 u + g
#pragma unroll
    for (int j = 1; j < 4; ++j)
      if (g == j) mine = sbyte[4 * u + j];
    sb[u] = mine;
  }
}

template <typename T>
__device__ __forceinline__ void col_load(const T *__restrict__ src, int64_t cols, int64_t c, int64_t r0, bool live,
                                         int g, uint4 (&w)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i)
    w[i] = live ? __ldcs(reinterpret_cast<const uint4 *>(src + (r0 + g + 4 * i) * cols + c)) : make_uint4(0, 0, 0, 0);
}

// A list of matrices for one launch of the warp-tile kernel: one call's matrix, or a
// group of columnwise views quantized together.  The blocks of every matrix form one 1-D
// grid, matrix after matrix; within a matrix, blocks run across the columns first.
constexpr int kColItems = 8;
constexpr int kColStripsTile = 2;  // 32-row strips a warp takes, one after the other
struct ColItem {
  const void *src;
  uint8_t *qt, *st;
  int64_t rows, cols;
  int64_t sf_words;     // 0: scales [cols, rows / 32]; else the tiled layout's words a row
  int32_t bf16;         // source element type: bf16, else fp32
  int32_t pack;         // a warp's scale bytes of a column go out as one store
  int32_t gx;           // blocks across the columns
  int32_t block_begin;  // this matrix's first block in the grid
};
struct ColArgs {
  ColItem it[kColItems];
  int32_t n;
};

// Block (bx, by) of one matrix: its warps take adjacent column tiles of 8 x VE columns and
// the strips S by .. S by + S - 1 of them.
template <typename T, int S>
__device__ __forceinline__ void col_tile_block(const ColItem &it, int bx, int by) {
  constexpr int VE = ColTile<T>::VE, NQ = VE / 4;
  const T *__restrict__ src = static_cast<const T *>(it.src);
  const int64_t rows = it.rows, cols = it.cols;
  const int lane = threadIdx.x & 31, g = lane >> 3, q = lane & 7;
  const int64_t c = (int64_t(bx) * (kColTileThreads / 32) + (threadIdx.x >> 5)) * (8 * VE) + VE * q;
  if (c - VE * q >= cols) return;  // the whole warp is past the last column
  const bool live = c < cols;      // cols % VE == 0: a lane's columns are all in or all out
  const int64_t strips = rows / 32;
  const int64_t s0 = int64_t(by) * S;
  uint32_t sc[NQ] = {};  // the scale bytes of column 4 u + g, strip s at byte s
#pragma unroll 1
  for (int s = 0; s < S; ++s) {
    if (s0 + s >= strips) break;
    const int64_t r0 = (s0 + s) * 32;
    uint4 w[8];
    col_load(src, cols, c, r0, live, g, w);
    uint32_t sb[NQ];
    col_unit<T>(w, it.qt, rows, c, r0, live, g, sb);
#pragma unroll
    for (int u = 0; u < NQ; ++u) sc[u] |= sb[u] << (8 * s);
  }
  if (!live) return;
  const int ns = int(strips - s0 < S ? strips - s0 : S);
#pragma unroll
  for (int u = 0; u < NQ; ++u) {
    if (it.pack && ns == S) {  // the S bytes are adjacent in either layout (s0 a multiple of S)
      uint8_t *p = it.st + scale_index_rc(c + 4 * u + g, s0, strips, it.sf_words);
      if (S == 4) *reinterpret_cast<uint32_t *>(p) = sc[u];
      else if (S == 2) *reinterpret_cast<uint16_t *>(p) = uint16_t(sc[u]);
      else *p = uint8_t(sc[u]);
    } else {
      for (int s = 0; s < ns; ++s)
        it.st[scale_index_rc(c + 4 * u + g, s0 + s, strips, it.sf_words)] = uint8_t(sc[u] >> (8 * s));
    }
  }
}

__global__ void __launch_bounds__(kColTileThreads) mx_quantize_col_tile_kernel(const __grid_constant__ ColArgs a) {
  gtp::ptx::allow_dependents();
  gtp::ptx::wait_prior_grid();
  const int b = int(blockIdx.x);
  int i = 0;
  while (i + 1 < a.n && b >= a.it[i + 1].block_begin) ++i;
  const ColItem &it = a.it[i];
  const int local = b - it.block_begin;
  const int by = local / it.gx, bx = local - by * it.gx;
  if (it.bf16) col_tile_block<__nv_bfloat16, kColStripsTile>(it, bx, by);
  else col_tile_block<float, kColStripsTile>(it, bx, by);
}

// Whether the warp-tile kernel takes a matrix: every source row starts on 16 bytes (cols a
// multiple of the 16-byte vector, src 16-byte aligned).
bool col_tile_ok(const void *src, bool bf16, int64_t cols) {
  return cols % (bf16 ? ColTile<__nv_bfloat16>::VE : ColTile<float>::VE) == 0 && gtp::aligned16(src);
}

// One launch of the warp-tile kernel over items[0..n) (1 <= n <= kColItems, each non-empty
// and accepted by col_tile_ok).
gtp_status launch_col_tile(const ColItem *items, int n, cudaStream_t stream) {
  ColArgs a;
  std::memset(&a, 0, sizeof(a));
  int64_t blocks = 0;
  for (int i = 0; i < n; ++i) {
    ColItem &it = a.it[i];
    it = items[i];
    const int ve = it.bf16 ? ColTile<__nv_bfloat16>::VE : ColTile<float>::VE;
    const int64_t strips = it.rows / 32;
    const int64_t block_cols = (kColTileThreads / 32) * 8 * ve;  // a column tile a warp
    it.gx = int32_t((it.cols + block_cols - 1) / block_cols);
    it.pack = it.sf_words ? 1
                          : (strips % kColStripsTile == 0 && reinterpret_cast<uintptr_t>(it.st) % kColStripsTile == 0)
                              ? 1
                              : 0;
    it.block_begin = int32_t(blocks);
    blocks += int64_t(it.gx) * ((strips + kColStripsTile - 1) / kColStripsTile);
    if (blocks > INT32_MAX) return gtp::fail(GTP_E_SHAPE, "too many blocks in one launch");
  }
  a.n = n;
  return gtp::launch_overlapped(mx_quantize_col_tile_kernel, unsigned(blocks), kColTileThreads, 0, stream,
                                "mxfp8_quantize_columnwise", a);
}

// tiled: the scales in the tiled layout (gtp_sf_tile of the [cols, rows / 32] array)
ColItem col_item(const void *src, bool bf16, int64_t rows, int64_t cols, uint8_t *qt, uint8_t *st, bool tiled) {
  ColItem it{};
  it.src = src;
  it.qt = qt;
  it.st = st;
  it.rows = rows;
  it.cols = cols;
  it.sf_words = tiled ? (rows / 32 + 3) / 4 : 0;
  it.bf16 = bf16 ? 1 : 0;
  return it;
}

template <typename T>
gtp_status launch_col_strip(const T *src, int64_t rows, int64_t cols, uint8_t *qt, uint8_t *st, int64_t words,
                            cudaStream_t stream) {
  if (cols % 2 == 0 && reinterpret_cast<uintptr_t>(src) % (2 * sizeof(T)) == 0)
    return launch_col_v<T, 2>(src, rows, cols, qt, st, words, stream);
  return launch_col_v<T, 1>(src, rows, cols, qt, st, words, stream);
}

// The strip kernel for one matrix (a matrix the warp-tile kernel does not take, or all of
// them when GTP_MXCOL_VARIANT = "strip", for measurements).
gtp_status launch_col_strip_any(const void *src, bool bf16, int64_t rows, int64_t cols, uint8_t *qt, uint8_t *st,
                                bool tiled, cudaStream_t stream) {
  const int64_t words = tiled ? (rows / 32 + 3) / 4 : 0;
  if (bf16) return launch_col_strip(static_cast<const __nv_bfloat16 *>(src), rows, cols, qt, st, words, stream);
  return launch_col_strip(static_cast<const float *>(src), rows, cols, qt, st, words, stream);
}

bool col_strip_forced() {
  const char *v = std::getenv("GTP_MXCOL_VARIANT");
  return v && std::strcmp(v, "strip") == 0;
}

// The arguments of one columnwise quantization, as the single entry point checks them.
gtp_status check_col(const void *src, int32_t src_dt, int64_t rows, int64_t cols, const uint8_t *e4m3_t,
                     const uint8_t *e8m0_t, bool tiled) {
  if (src_dt != GTP_F32 && src_dt != GTP_BF16) return gtp::fail(GTP_E_DTYPE, "src must be F32 or BF16");
  if (rows < 0 || cols < 0) return gtp::fail(GTP_E_ARG, "negative size");
  if (rows % 32) return gtp::fail(GTP_E_SHAPE, "rows must be a multiple of 32");
  if (cols > (int64_t(1) << 31) || rows > (int64_t(1) << 36) / (cols ? cols : 1))
    return gtp::fail(GTP_E_SHAPE, "matrix too large");
  if (rows == 0 || cols == 0) return GTP_OK;
  if (!src || !e4m3_t || !e8m0_t) return gtp::fail(GTP_E_ARG, "null pointer");
  if (!gtp::aligned16(e4m3_t)) return gtp::fail(GTP_E_ALIGN, "e4m3_t must be 16-byte aligned");
  if (tiled && !gtp::aligned16(e8m0_t)) return gtp::fail(GTP_E_ALIGN, "tiled scales must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(src) & (src_dt == GTP_F32 ? 3u : 1u)) return gtp::fail(GTP_E_ALIGN, "src alignment");
  if (rows / 32 > 65535) return gtp::fail(GTP_E_SHAPE, "rows / 32 above 65535");
  return GTP_OK;
}

}  // namespace

namespace {
gtp_status quantize_columnwise(const void *src, gtp_dtype src_dt, int64_t rows, int64_t cols, uint8_t *e4m3_t,
                               uint8_t *e8m0_t, bool tiled, gtp_stream stream) {
  if (gtp_status s = check_col(src, src_dt, rows, cols, e4m3_t, e8m0_t, tiled)) return s;
  if (rows == 0 || cols == 0) return GTP_OK;
  gtp::DeviceInfo dev;
  if (gtp_status s = gtp::require_sm103(&dev)) return s;
  cudaStream_t st = gtp::as_stream(stream);
  const bool bf16 = src_dt == GTP_BF16;
  if (col_tile_ok(src, bf16, cols) && !col_strip_forced()) {
    const ColItem it = col_item(src, bf16, rows, cols, e4m3_t, e8m0_t, tiled);
    return launch_col_tile(&it, 1, st);
  }
  return launch_col_strip_any(src, bf16, rows, cols, e4m3_t, e8m0_t, tiled, st);
}
}  // namespace

extern "C" gtp_status gtp_mxfp8_quantize_columnwise(const void *src, gtp_dtype src_dt, int64_t rows, int64_t cols,
                                                    uint8_t *e4m3_t, uint8_t *e8m0_t, gtp_stream stream) {
  gtp::clear_error();
  return quantize_columnwise(src, src_dt, rows, cols, e4m3_t, e8m0_t, false, stream);
}

extern "C" gtp_status gtp_mxfp8_quantize_columnwise_tiled(const void *src, gtp_dtype src_dt, int64_t rows,
                                                          int64_t cols, uint8_t *e4m3_t, uint8_t *e8m0_t_tiled,
                                                          gtp_stream stream) {
  gtp::clear_error();
  return quantize_columnwise(src, src_dt, rows, cols, e4m3_t, e8m0_t_tiled, true, stream);
}

namespace {

// The bytes a group reads (sources) and writes (codes, scales): an output that overlaps a
// source or another output is an argument error, found before anything is launched (the
// launch would race on those bytes).  Sources may overlap each other.
struct ByteRange {
  uintptr_t lo, hi;
  int desc;
  const char *what;  // nullptr: a source
};

void add_range(ByteRange *r, int &nr, const void *p, int64_t bytes, int desc, const char *what) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  r[nr++] = ByteRange{lo, lo + uintptr_t(bytes), desc, what};
}

gtp_status check_group_overlaps(const ByteRange *r, int nr) {
  for (int i = 0; i < nr; ++i)
    for (int j = i + 1; j < nr; ++j)
      if ((r[i].what || r[j].what) && r[i].lo < r[j].hi && r[j].lo < r[i].hi)
        return gtp::fail(GTP_E_ARG, "descriptor %d's %s overlaps descriptor %d's %s", r[i].desc,
                         r[i].what ? r[i].what : "source", r[j].desc, r[j].what ? r[j].what : "source");
  return GTP_OK;
}

}  // namespace

extern "C" gtp_status gtp_mxfp8_quantize_columnwise_group(const gtp_mx_col_desc *descs, int32_t n,
                                                          gtp_stream stream) {
  gtp::clear_error();
  if (n < 0 || n > kColItems) return gtp::fail(GTP_E_ARG, "n must lie in [0, %d]", kColItems);
  if (n > 0 && !descs) return gtp::fail(GTP_E_ARG, "null descriptor array");
  for (int i = 0; i < n; ++i) {  // every argument is checked before anything is launched
    const gtp_mx_col_desc &d = descs[i];
    if (d.tiled_scales != 0 && d.tiled_scales != 1)
      return gtp::fail(GTP_E_ARG, "descriptor %d: tiled_scales must be 0 or 1", i);
    if (gtp_status s = check_col(d.src, d.src_dtype, d.rows, d.cols, d.e4m3_t, d.e8m0_t, d.tiled_scales != 0))
      return s;
  }
  ByteRange ranges[3 * kColItems];
  int nr = 0;
  for (int i = 0; i < n; ++i) {
    const gtp_mx_col_desc &d = descs[i];
    if (d.rows == 0 || d.cols == 0) continue;
    add_range(ranges, nr, d.src, d.rows * d.cols * (d.src_dtype == GTP_BF16 ? 2 : 4), i, nullptr);
    add_range(ranges, nr, d.e4m3_t, d.rows * d.cols, i, "codes");
    add_range(ranges, nr, d.e8m0_t, d.tiled_scales ? gtp_sf_tiled_bytes(d.cols, d.rows / 32) : d.cols * (d.rows / 32),
              i, "scales");
  }
  if (gtp_status s = check_group_overlaps(ranges, nr)) return s;
  ColItem tiles[kColItems];
  int ntiles = 0, nstrips = 0;
  const bool strip = col_strip_forced();
  for (int i = 0; i < n; ++i) {
    const gtp_mx_col_desc &d = descs[i];
    if (d.rows == 0 || d.cols == 0) continue;
    const bool bf16 = d.src_dtype == GTP_BF16;
    if (col_tile_ok(d.src, bf16, d.cols) && !strip)
      tiles[ntiles++] = col_item(d.src, bf16, d.rows, d.cols, d.e4m3_t, d.e8m0_t, d.tiled_scales != 0);
    else ++nstrips;
  }
  if (ntiles + nstrips == 0) return GTP_OK;
  gtp::DeviceInfo dev;
  if (gtp_status s = gtp::require_sm103(&dev)) return s;
  cudaStream_t st = gtp::as_stream(stream);
  for (int i = 0; i < n && nstrips > 0; ++i) {  // matrices the warp-tile kernel does not take: launches of their own
    const gtp_mx_col_desc &d = descs[i];
    if (d.rows == 0 || d.cols == 0) continue;
    const bool bf16 = d.src_dtype == GTP_BF16;
    if (col_tile_ok(d.src, bf16, d.cols) && !strip) continue;
    if (gtp_status s = launch_col_strip_any(d.src, bf16, d.rows, d.cols, d.e4m3_t, d.e8m0_t, d.tiled_scales != 0, st))
      return s;
  }
  return ntiles ? launch_col_tile(tiles, ntiles, st) : GTP_OK;
}

namespace {

// The arguments of one rowwise quantization.
gtp_status check_row(const void *src, int32_t src_dt, int64_t rows, int64_t cols, const uint8_t *e4m3,
                     const uint8_t *e8m0) {
  if (src_dt != GTP_F32 && src_dt != GTP_BF16) return gtp::fail(GTP_E_DTYPE, "src must be F32 or BF16");
  if (rows < 0 || cols < 0) return gtp::fail(GTP_E_ARG, "negative size");
  if (cols % 32) return gtp::fail(GTP_E_SHAPE, "cols must be a multiple of 32");
  if (rows > (int64_t(1) << 40) / (cols ? cols : 1)) return gtp::fail(GTP_E_SHAPE, "matrix too large");
  if (rows == 0 || cols == 0) return GTP_OK;
  if (!src || !e4m3 || !e8m0) return gtp::fail(GTP_E_ARG, "null pointer");
  if (!gtp::aligned16(src) || !gtp::aligned16(e4m3)) return gtp::fail(GTP_E_ALIGN, "src and e4m3 must be 16-byte aligned");
  return GTP_OK;
}

gtp_status quantize_rowwise(const void *src, gtp_dtype src_dt, int64_t rows, int64_t cols, uint8_t *e4m3,
                            uint8_t *e8m0, bool tiled, gtp_stream stream) {
  gtp::clear_error();
  if (gtp_status s = check_row(src, src_dt, rows, cols, e4m3, e8m0)) return s;
  if (rows == 0 || cols == 0) return GTP_OK;
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

extern "C" gtp_status gtp_mxfp8_quantize_rowwise_group(const gtp_mx_row_desc *descs, int32_t n, gtp_stream stream) {
  gtp::clear_error();
  if (n < 0 || n > kRowItems) return gtp::fail(GTP_E_ARG, "n must lie in [0, %d]", kRowItems);
  if (n > 0 && !descs) return gtp::fail(GTP_E_ARG, "null descriptor array");
  RowArgs a;
  std::memset(&a, 0, sizeof(a));
  int64_t total = 0;
  for (int i = 0; i < n; ++i) {  // every argument is checked before anything is launched
    const gtp_mx_row_desc &d = descs[i];
    if (d.tiled_scales != 0 && d.tiled_scales != 1)
      return gtp::fail(GTP_E_ARG, "descriptor %d: tiled_scales must be 0 or 1", i);
    if (gtp_status s = check_row(d.src, d.src_dtype, d.rows, d.cols, d.e4m3, d.e8m0)) return s;
    if (d.rows == 0 || d.cols == 0) continue;
    RowItem &it = a.it[a.n++];
    it.src = d.src;
    it.q = d.e4m3;
    it.scale = d.e8m0;
    it.nvec = d.rows * d.cols / 8;
    it.C = d.cols / 32;
    it.words = d.tiled_scales ? (it.C + 3) / 4 : 0;
    it.bf16 = d.src_dtype == GTP_BF16;
    total += it.nvec;
  }
  if (a.n == 0) return GTP_OK;
  ByteRange ranges[3 * kRowItems];
  int nr = 0;
  for (int i = 0; i < n; ++i) {
    const gtp_mx_row_desc &d = descs[i];
    if (d.rows == 0 || d.cols == 0) continue;
    add_range(ranges, nr, d.src, d.rows * d.cols * (d.src_dtype == GTP_BF16 ? 2 : 4), i, nullptr);
    add_range(ranges, nr, d.e4m3, d.rows * d.cols, i, "codes");
    add_range(ranges, nr, d.e8m0, d.tiled_scales ? gtp_sf_tiled_bytes(d.rows, d.cols / 32) : d.rows * (d.cols / 32), i,
              "scales");
  }
  if (gtp_status s = check_group_overlaps(ranges, nr)) return s;
  gtp::DeviceInfo dev;
  if (gtp_status s = gtp::require_sm103(&dev)) return s;
  const int64_t want = (total + kThreads - 1) / kThreads;
  const int grid = int(std::max<int64_t>(1, std::min<int64_t>(want, int64_t(dev.sm_count) * 8)));
  return gtp::launch_overlapped(mx_quantize_group_kernel, grid, kThreads, 0, gtp::as_stream(stream),
                                "mxfp8_quantize_rowwise", a);
}

extern "C" gtp_status gtp_mxfp8_quantize_rowwise_tiled(const void *src, gtp_dtype src_dt, int64_t rows, int64_t cols,
                                                       uint8_t *e4m3, uint8_t *e8m0_tiled, gtp_stream stream) {
  return quantize_rowwise(src, src_dt, rows, cols, e4m3, e8m0_tiled, true, stream);
}
