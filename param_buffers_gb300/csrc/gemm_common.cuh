// Pieces shared by the tensor-core GEMM kernels: the bf16 GEMMs (gemm_bf16.cu) and the
// block-scaled MXFP8 / NVFP4 GEMMs (gemm_blockscaled.cu).  Everything here has internal
// linkage, so each translation unit holds its own copy, including its own wait-timeout
// word (a device variable cannot be shared between units compiled without relocatable
// device code).
#pragma once
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>

#include "device.h"
#include "sm100_ptx.cuh"
#include "tensor_map.h"

namespace gtp {
gtp_status launch_zero_bytes(void *data, int64_t nbytes, cudaStream_t stream, int sm_count);
void clear_error();
}

namespace {

using namespace gtp::ptx;

// Bits of kernel wait timeouts of this translation unit (see gtp_wait_timeouts).
__device__ unsigned int g_gtp_wait_timeouts;

constexpr int BM = 128, BN = 256, BK = 64, UK = 16;
constexpr int STAGES = 4;
constexpr int kGemmThreads = 192;
constexpr int A_STAGE = BM * BK * 2;  // 16 KB
constexpr int B_STAGE = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_STAGE + B_STAGE;
constexpr int EPI_WARPS = 4;
constexpr int EPI_BUF = 32 * 128;  // 32 rows x 128 bytes
constexpr int SMEM_OPERANDS = STAGES * STAGE_BYTES;
constexpr int SMEM_EPI = EPI_WARPS * 2 * EPI_BUF;
constexpr int SMEM_CTRL = 256;
constexpr int SMEM_TOTAL = SMEM_OPERANDS + SMEM_EPI + SMEM_CTRL + 1024;  // + alignment slack
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr int MN_CHUNK = 64 * BK * 2;  // one 64-wide MN-major box: 64 K rows of 128 bytes
static_assert(SMEM_TOTAL <= 232448, "shared memory per block");

// Epilogues: a bf16 store and an fp32 reduce-add, both by TMA from swizzled staging; and,
// for main_grad views that TMA cannot address (a start that is not 16-byte aligned, or a
// bf16 buffer), two that write from registers: fp32 atomic adds (kReduceAddF32Direct) and a
// bf16 read-add-round-write (kAccumBf16; one CTA owns each element, no split contraction).
enum { kStoreBf16 = 0, kReduceAddF32 = 1, kReduceAddF32Direct = 2, kAccumBf16 = 3 };

__host__ __device__ constexpr bool epi_by_tma(int epi) { return epi == kStoreBf16 || epi == kReduceAddF32; }

// Division of 0 <= n < 2^31 by a fixed d >= 1 as one multiply and a shift (the round-up
// method of Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994): with l = ceil(log2 d) and m = ceil(2^(31+l) / d) < 2^32,
// floor(n / d) = (n m) >> (31 + l).  The unit decode below runs once per tile in every
// warp role; with hardware division (two of them 64-bit) it cost about 1000 cycles.
struct FastDiv {
  uint32_t m, s;
};

inline FastDiv make_fastdiv(int d) {
  uint32_t l = 0;
  while ((uint64_t(1) << l) < uint64_t(d)) ++l;
  const uint64_t num = uint64_t(1) << (31 + l);
  return {uint32_t((num + uint64_t(d) - 1) / uint64_t(d)), 31 + l};
}

__device__ __forceinline__ int fast_div(int n, FastDiv f) {
  return int((uint64_t(uint32_t(n)) * f.m) >> f.s);
}

struct Problem {
  int32_t m_dim, n_dim, k_dim;  // D rows, D columns, contraction length
  int32_t tiles_m, tiles_n, k_blocks, splits, num_units, group_m;
  // derived by finalize_problem: tiles per group of group_m tile rows, the last group
  // (which may hold fewer tile rows) and its height, and the divisions the decode needs
  int32_t per_group, last_group, gm_last;
  FastDiv f_splits, f_per_group, f_gm, f_gm_last;
  // half-width tail (CTA-pair bf16 GEMM only): units from tail_first on are the 128-column
  // halves of tiles tail_first, tail_first + 1, ... (two units a tile)
  int32_t tail_first, tail_half;
  // L2 cache policy of the A and B operand loads (CTA-pair bf16 GEMM): 0 normal,
  // 1 evict_first, 2 evict_last
  int32_t hint_a, hint_b;
  // the output (D, n_dim elements a row) for the epilogues that write from registers
  void *direct;
};

// Fills the derived fields once splits, group_m and the tile counts are set; every
// (split + 1) * k_blocks stays below 2^31 (at most 8 splits, k_blocks <= 2^24).
inline void finalize_problem(Problem &p) {
  p.tail_first = p.num_units;
  p.tail_half = 0;
  p.hint_a = p.hint_b = 0;
  p.per_group = p.group_m * p.tiles_n;
  p.last_group = (p.tiles_m - 1) / p.group_m;
  p.gm_last = p.tiles_m - p.last_group * p.group_m;
  p.f_splits = make_fastdiv(p.splits);
  p.f_per_group = make_fastdiv(p.per_group);
  p.f_gm = make_fastdiv(p.group_m);
  p.f_gm_last = make_fastdiv(p.gm_last);
}

// Unit u -> output tile (tm, tn) and its k-block range [kb0, kb1).  Units enumerate
// (tile, split) pairs with the split fastest; tiles go in groups of group_m tile rows,
// column-major inside a group, so that CTAs running at the same time share operand tiles
// in L2.
__device__ __forceinline__ void decode_unit(const Problem &p, int u, int &tm, int &tn, int &kb0, int &kb1) {
  const int t = fast_div(u, p.f_splits);
  const int split = u - t * p.splits;
  const int g = fast_div(t, p.f_per_group);
  const bool last = g == p.last_group;
  const int gm = last ? p.gm_last : p.group_m;
  const int r = t - g * p.per_group;
  const int q = fast_div(r, last ? p.f_gm_last : p.f_gm);
  tm = g * p.group_m + (r - q * gm);
  tn = q;
  kb0 = fast_div(split * p.k_blocks, p.f_splits);
  kb1 = fast_div((split + 1) * p.k_blocks, p.f_splits);
}

// decode_unit, plus which 128-column half of the tile a half-width tail unit covers (-1
// for a whole tile).  Tail units exist only without split contractions.
__device__ __forceinline__ void decode_unit_half(const Problem &p, int u, int &tm, int &tn, int &kb0, int &kb1,
                                                 int &half) {
  half = -1;
  if (p.tail_half && u >= p.tail_first) {
    const int v = u - p.tail_first;
    half = v & 1;
    u = p.tail_first + (v >> 1);
  }
  decode_unit(p, u, tm, tn, kb0, kb1);
}

// A wait that ignores the abort flag: used to drain this CTA's own asynchronous work.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(&g_gtp_wait_timeouts, 0x80u);
      return;
    }
  }
}


// Writes one 32-row x 128-byte chunk of a warp's accumulator rows into swizzled staging
// shared memory (the 128-byte swizzle the output tensor map uses): bf16 takes 64 fp32
// columns (r0, r1), fp32 takes 32 (r0).  Row `lane`, 16-byte chunk j goes to j ^ (lane % 8).
template <int EPI>
__device__ __forceinline__ void stage_rows(uint8_t *buf, int lane, const uint32_t (&r0)[32], const uint32_t (&r1)[32]) {
  uint8_t *rowp = buf + lane * 128;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint4 v;
    if (EPI == kStoreBf16) {
      uint32_t w[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int e = 8 * j + 2 * h;  // columns e, e+1 of this chunk
        const float lo = __uint_as_float(e < 32 ? r0[e] : r1[e - 32]);
        const float hi = __uint_as_float(e + 1 < 32 ? r0[e + 1] : r1[e + 1 - 32]);
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
        w[h] = *reinterpret_cast<const uint32_t *>(&b2);
      }
      v = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      v = make_uint4(r0[4 * j], r0[4 * j + 1], r0[4 * j + 2], r0[4 * j + 3]);
    }
    *reinterpret_cast<uint4 *>(rowp + ((j ^ (lane & 7)) << 4)) = v;
  }
}

// The same for a 32-row x 64-byte chunk under the 64-byte swizzle: bf16 takes 32 columns
// (c0 .. c0 + 31 of r), fp32 16.  Row `lane`, 16-byte chunk j goes to j ^ ((lane / 2) % 4).
template <int EPI>
__device__ __forceinline__ void stage_rows64(uint8_t *buf, int lane, const uint32_t (&r)[32], int c0) {
  uint8_t *rowp = buf + lane * 64;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint4 v;
    if (EPI == kStoreBf16) {
      uint32_t w[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(r[8 * j + 2 * h]),
                                                        __uint_as_float(r[8 * j + 2 * h + 1]));
        w[h] = *reinterpret_cast<const uint32_t *>(&b2);
      }
      v = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      v = make_uint4(r[c0 + 4 * j], r[c0 + 4 * j + 1], r[c0 + 4 * j + 2], r[c0 + 4 * j + 3]);
    }
    *reinterpret_cast<uint4 *>(rowp + ((j ^ ((lane >> 1) & 3)) << 4)) = v;
  }
}

// The register epilogues.  Lane l of an epilogue warp holds row `row` (its own) of a chunk
// of the accumulator: columns col .. col + 31 in r (fp32 bits).  Rows of D are n_dim
// elements long and n_dim % 8 == 0, so every row of a view starts with the same alignment
// as its first: H leading elements up to a 16-byte boundary, then aligned groups of four.
template <int H>
__device__ __forceinline__ void red_row_f32_h(float *p, int n, const uint32_t (&r)[32]) {
#pragma unroll
  for (int j = 0; j < H; ++j)
    if (j < n) atomicAdd(p + j, __uint_as_float(r[j]));
#pragma unroll
  for (int q = 0; q < (32 - H) / 4; ++q) {
    const int j = H + 4 * q;
    if (j + 3 < n) {
      atomicAdd(reinterpret_cast<float4 *>(p + j), make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                                                __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3])));
    } else {
#pragma unroll
      for (int t = 0; t < 4; ++t)
        if (j + t < n) atomicAdd(p + j + t, __uint_as_float(r[j + t]));
    }
  }
#pragma unroll
  for (int j = H + 4 * ((32 - H) / 4); j < 32; ++j)
    if (j < n) atomicAdd(p + j, __uint_as_float(r[j]));
}

// D[row, col .. col + 31] += r (fp32 atomic adds; the view may start at any element).
__device__ __forceinline__ void red_row_f32(void *d, int row, int col, int m_dim, int n_dim, const uint32_t (&r)[32]) {
  if (row >= m_dim || col >= n_dim) return;
  float *p = static_cast<float *>(d) + int64_t(row) * n_dim + col;
  const int n = min(32, n_dim - col);
  switch (int((16u - (uint32_t(reinterpret_cast<uintptr_t>(p)) & 15u)) & 15u) >> 2) {
    case 0: red_row_f32_h<0>(p, n, r); break;
    case 1: red_row_f32_h<1>(p, n, r); break;
    case 2: red_row_f32_h<2>(p, n, r); break;
    default: red_row_f32_h<3>(p, n, r); break;
  }
}

// D[row, col .. col + 63] = RNE_bf16(D + acc) for a bf16 D, acc = r0 (columns 0-31) and r1
// (32-63): one rounding of the fp32 sum, as an fp32-computed accumulate into a bf16 buffer.
__device__ __forceinline__ void accum_row_bf16(void *d, int row, int col, int m_dim, int n_dim,
                                               const uint32_t (&r0)[32], const uint32_t (&r1)[32]) {
  if (row >= m_dim || col >= n_dim) return;
  __nv_bfloat16 *p = static_cast<__nv_bfloat16 *>(d) + int64_t(row) * n_dim + col;
  const int n = min(64, n_dim - col);  // a multiple of 8
  if ((reinterpret_cast<uintptr_t>(p) & 15u) == 0) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (8 * q < n) {
        uint4 v = *reinterpret_cast<const uint4 *>(p + 8 * q);
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int e = 8 * q + 2 * h;
          const __nv_bfloat162 old = *reinterpret_cast<const __nv_bfloat162 *>(&w[h]);
          const float a0 = __uint_as_float(e < 32 ? r0[e] : r1[e - 32]);
          const float a1 = __uint_as_float(e + 1 < 32 ? r0[e + 1] : r1[e + 1 - 32]);
          const __nv_bfloat162 nw = __floats2bfloat162_rn(__low2float(old) + a0, __high2float(old) + a1);
          w[h] = *reinterpret_cast<const uint32_t *>(&nw);
        }
        *reinterpret_cast<uint4 *>(p + 8 * q) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < 64; ++e)
      if (e < n) p[e] = __float2bfloat16_rn(__bfloat162float(p[e]) + __uint_as_float(e < 32 ? r0[e] : r1[e - 32]));
  }
}

// Split count of a reduce-add GEMM: the wave occupancy of its units less 0.06 per extra
// split (each split reduce-adds one more fp32 copy of the output).  Measured on the layer
// wgrads (pair kernel), the per-shape best: fc2 1 (84.3 us against 89.3 with 4 splits),
// fc1 2, QKV 3, O projection 2; a 0.03 charge had picked 4 for fc2.
int choose_splits(int tiles, int k_blocks, int sms) {
  int best = 1;
  double best_score = -1.0;
  for (int s = 1; s <= 8 && s <= k_blocks; ++s) {
    if (s > 1 && k_blocks / s < 4) break;
    const int64_t units = int64_t(tiles) * s;
    const int64_t waves = (units + sms - 1) / sms;
    const double score = double(units) / double(waves * sms) - 0.06 * (s - 1);
    if (score > best_score + 1e-9) {
      best_score = score;
      best = s;
    }
  }
  return best;
}

using CU = CUtensorMapDataType;
constexpr CU kBF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
constexpr CU kF32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
constexpr CUtensorMapSwizzle kSW128 = CU_TENSOR_MAP_SWIZZLE_128B;

template <typename K>
gtp_status configure(K kernel, int smem, std::atomic<uint64_t> &configured, int device) {
  const uint64_t bit = uint64_t(1) << (device & 63);
  if (configured.load() & bit) return GTP_OK;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return gtp::fail(GTP_E_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  configured.fetch_or(bit);
  return GTP_OK;
}

constexpr int64_t kMaxDim = int64_t(1) << 30;

}  // namespace
