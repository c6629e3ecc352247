// The local fp32 sum of the all-to-all reduce-scatter.
//
// Page: "05 · grad/param buffer: contiguous buffer data structures and read/write loop"
// (llm-infra-atlas) §9.1, reduce_scatter_with_fp32_accumulation: the bucket's
// reduce-scatter is an all-to-all in which every rank receives the world_size
// low-precision slices of its own shard; when the exchange completes the rank adds them
// up with an fp32 sum and casts the total back to the output's dtype.  This is that sum,
// on the GPU that holds the received slices: out[i] = cast(slice_0[i] + ... + slice_{P-1}[i]),
// accumulated in fp32 in rank order, one rounding per addition (the reading of the
// oracle), and rounded once (to nearest even) to a bf16 output.
//
// Memory-bound: P x (2 or 4) bytes read and 2 or 4 written per element.  A rank's shard
// is short (1M elements for the 7B buffer at dp 64) and the slices many, and the rank-order
// sum is a chain per element: the slices' pieces of a chunk are staged in shared memory
// first, so that the loads of all P slices are in flight together.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cstring>

#include "device.h"
#include "sm100_ptx.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kMaxSlices = 128;

struct RsArgs {
  const void *slice[kMaxSlices];
  void *out;
  int64_t n;
  int32_t P;
  int32_t in_bf16, out_bf16;  // the launch picks the kernel instance from these
};

// A block takes a chunk of E consecutive elements: it copies every slice's piece of the
// chunk into shared memory with asynchronous 16-byte copies (all of them in flight at
// once, no registers held), then each of the chunk's 16-byte units is summed over the
// slices in rank order by one thread, from shared memory.  E is chosen so that the P
// pieces fit 24 KB: small chunks make many blocks, so the SMs stay evenly loaded on a
// short shard and one block's copies overlap another's additions (64 slices of a
// 1M-element bf16 shard: 5.45 TB/s with 24 KB, 5.28 with 32, 4.33 with 64, 4.00 with 96).
constexpr int kStageBytes = 24 * 1024;

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(gtp::ptx::smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// 16 bytes of elements as fp32: 8 bf16 or 4 fp32.
template <bool IN_BF16>
__device__ __forceinline__ void unpack(const uint4 w, float (&x)[IN_BF16 ? 8 : 4]) {
  if constexpr (IN_BF16) {
    x[0] = __uint_as_float(w.x << 16); x[1] = __uint_as_float(w.x & 0xFFFF0000u);
    x[2] = __uint_as_float(w.y << 16); x[3] = __uint_as_float(w.y & 0xFFFF0000u);
    x[4] = __uint_as_float(w.z << 16); x[5] = __uint_as_float(w.z & 0xFFFF0000u);
    x[6] = __uint_as_float(w.w << 16); x[7] = __uint_as_float(w.w & 0xFFFF0000u);
  } else {
    x[0] = __uint_as_float(w.x); x[1] = __uint_as_float(w.y); x[2] = __uint_as_float(w.z); x[3] = __uint_as_float(w.w);
  }
}

template <bool IN_BF16>
__device__ __forceinline__ float load1(const RsArgs &a, int s, int64_t i) {
  if constexpr (IN_BF16) return __uint_as_float(uint32_t(static_cast<const unsigned short *>(a.slice[s])[i]) << 16);
  else return static_cast<const float *>(a.slice[s])[i];
}

template <bool OUT_BF16>
__device__ __forceinline__ void store1(const RsArgs &a, int64_t i, float v) {
  if constexpr (OUT_BF16) static_cast<__nv_bfloat16 *>(a.out)[i] = __float2bfloat16_rn(v);
  else static_cast<float *>(a.out)[i] = v;
}

template <bool IN_BF16, bool OUT_BF16>
__global__ void __launch_bounds__(kThreads) rs_local_sum_kernel(const __grid_constant__ RsArgs a, int64_t chunk) {
  extern __shared__ __align__(16) uint8_t stage[];
  gtp::ptx::allow_dependents();
  gtp::ptx::wait_prior_grid();
  constexpr int EU = IN_BF16 ? 8 : 4;       // elements a 16-byte unit
  constexpr int ESZ = IN_BF16 ? 2 : 4;
  const int64_t e0 = int64_t(blockIdx.x) * chunk;
  const int64_t e1 = min(e0 + chunk, a.n);
  const int units = int((e1 - e0) / EU);    // whole 16-byte units of each slice's piece
  const int unit_stride = int(chunk / EU);  // units a slice's piece holds in shared memory
  // every slice's whole units: P x units copies over the block's threads
  for (int j = threadIdx.x; j < a.P * units; j += blockDim.x) {
    const int s = j / units, u = j - s * units;
    cp_async16(stage + (size_t(s) * unit_stride + u) * 16,
               static_cast<const uint8_t *>(a.slice[s]) + (e0 + int64_t(u) * EU) * ESZ);
  }
  cp_async_wait_all();
  __syncthreads();
  for (int u = threadIdx.x; u < units; u += blockDim.x) {
    float acc[EU];
    unpack<IN_BF16>(*reinterpret_cast<const uint4 *>(stage + size_t(u) * 16), acc);
    for (int s = 1; s < a.P; ++s) {
      float x[EU];
      unpack<IN_BF16>(*reinterpret_cast<const uint4 *>(stage + (size_t(s) * unit_stride + u) * 16), x);
#pragma unroll
      for (int k = 0; k < EU; ++k) acc[k] = __fadd_rn(acc[k], x[k]);
    }
    const int64_t e = e0 + int64_t(u) * EU;
    if constexpr (OUT_BF16) {
      uint32_t w[EU / 2];
#pragma unroll
      for (int k = 0; k < EU / 2; ++k) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * k], acc[2 * k + 1]);
        w[k] = *reinterpret_cast<const uint32_t *>(&h);
      }
      if constexpr (EU == 8) __stcs(reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) + e), make_uint4(w[0], w[1], w[2], w[3]));
      else __stcs(reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(a.out) + e), make_uint2(w[0], w[1]));
    } else {
#pragma unroll
      for (int k = 0; k < EU; k += 4)
        __stcs(reinterpret_cast<float4 *>(static_cast<float *>(a.out) + e + k), make_float4(acc[k], acc[k + 1], acc[k + 2], acc[k + 3]));
    }
  }
  // the chunk's last elements that do not fill a unit (only the last chunk has any)
  for (int64_t i = e0 + int64_t(units) * EU + threadIdx.x; i < e1; i += blockDim.x) {
    float acc = load1<IN_BF16>(a, 0, i);
    for (int s = 1; s < a.P; ++s) acc = __fadd_rn(acc, load1<IN_BF16>(a, s, i));
    store1<OUT_BF16>(a, i, acc);
  }
}

// One launch of an instance; its shared-memory limit is raised once per device.
template <bool IN_BF16, bool OUT_BF16>
gtp_status launch_rs(const RsArgs &a, int64_t chunk, int64_t blocks, size_t smem, int device, cudaStream_t st) {
  static std::atomic<uint64_t> configured{0};
  const uint64_t bit = uint64_t(1) << (device & 63);
  if (!(configured.load() & bit)) {
    const cudaError_t e = cudaFuncSetAttribute(rs_local_sum_kernel<IN_BF16, OUT_BF16>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, kStageBytes);
    if (e != cudaSuccess) return gtp::fail(GTP_E_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    configured.fetch_or(bit);
  }
  return gtp::launch_overlapped(rs_local_sum_kernel<IN_BF16, OUT_BF16>, unsigned(blocks), kThreads, smem, st,
                                "rs_local_sum", a, chunk);
}

}  // namespace

extern "C" gtp_status gtp_rs_local_sum_rows(const void *slices, int64_t row_bytes, int32_t P, int64_t n,
                                            gtp_dtype in_dt, void *out, gtp_dtype out_dt, gtp_stream stream) {
  gtp::clear_error();
  if (P < 1 || P > kMaxSlices) return gtp::fail(GTP_E_ARG, "P must lie in [1, %d]", kMaxSlices);
  if (!slices && n > 0) return gtp::fail(GTP_E_ARG, "null receive buffer");
  if (row_bytes < 0) return gtp::fail(GTP_E_ARG, "negative row stride");
  const int64_t esz = in_dt == GTP_BF16 ? 2 : in_dt == GTP_F32 ? 4 : 0;  // others: gtp_rs_local_sum's error
  if (P > 1 && n > 0 && esz && row_bytes < n * esz) return gtp::fail(GTP_E_ARG, "row stride below a row's bytes");
  const void *rows[kMaxSlices] = {};
  if (slices)
    for (int r = 0; r < P; ++r) rows[r] = static_cast<const uint8_t *>(slices) + int64_t(r) * row_bytes;
  return gtp_rs_local_sum(rows, P, n, in_dt, out, out_dt, stream);
}

extern "C" gtp_status gtp_rs_local_sum(const void *const *slices, int32_t P, int64_t n, gtp_dtype in_dt, void *out,
                                       gtp_dtype out_dt, gtp_stream stream) {
  gtp::clear_error();
  if (P < 1 || P > kMaxSlices) return gtp::fail(GTP_E_ARG, "P must lie in [1, %d]", kMaxSlices);
  if (n < 0) return gtp::fail(GTP_E_ARG, "n < 0");
  if ((in_dt != GTP_BF16 && in_dt != GTP_F32) || (out_dt != GTP_BF16 && out_dt != GTP_F32))
    return gtp::fail(GTP_E_DTYPE, "slices and output must be GTP_BF16 or GTP_F32");
  if (!slices) return gtp::fail(GTP_E_ARG, "null slice array");
  if (n == 0) return GTP_OK;
  const size_t in_b = in_dt == GTP_BF16 ? 2 : 4, out_b = out_dt == GTP_BF16 ? 2 : 4;
  if (!out) return gtp::fail(GTP_E_ARG, "null output");
  if (!gtp::aligned16(out)) return gtp::fail(GTP_E_ALIGN, "out must be 16-byte aligned");
  const uintptr_t o0 = reinterpret_cast<uintptr_t>(out), o1 = o0 + size_t(n) * out_b;
  RsArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int s = 0; s < P; ++s) {
    if (!slices[s]) return gtp::fail(GTP_E_ARG, "slice %d is null", s);
    if (!gtp::aligned16(slices[s])) return gtp::fail(GTP_E_ALIGN, "slice %d must be 16-byte aligned", s);
    // the output may be one of the slices exactly (each element is read before it is
    // written, by the same thread), but not overlap one partly
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(slices[s]), s1 = s0 + size_t(n) * in_b;
    if (s0 < o1 && o0 < s1 && !(s0 == o0 && in_b == out_b))
      return gtp::fail(GTP_E_ARG, "out overlaps slice %d other than exactly", s);
    a.slice[s] = slices[s];
  }
  a.out = out;
  a.n = n;
  a.P = P;
  a.in_bf16 = in_dt == GTP_BF16;
  a.out_bf16 = out_dt == GTP_BF16;
  gtp::DeviceInfo dev;
  if (gtp_status s = gtp::require_sm103(&dev)) return s;
  // chunk: as many elements as keep the P pieces within kStageBytes, whole 16-byte units,
  // at most one unit per thread
  const int64_t per_unit = 16 / int64_t(in_b);
  int64_t units = std::min<int64_t>(kThreads, kStageBytes / (16 * int64_t(P)));
  units = std::max<int64_t>(units, 1);
  const int64_t chunk = units * per_unit;
  const size_t smem = size_t(P) * size_t(units) * 16;
  const int64_t blocks = (n + chunk - 1) / chunk;
  if (blocks > INT32_MAX) return gtp::fail(GTP_E_SHAPE, "n too large");
  cudaStream_t st = gtp::as_stream(stream);
  if (a.in_bf16 && a.out_bf16) return launch_rs<true, true>(a, chunk, blocks, smem, dev.device, st);
  if (a.in_bf16) return launch_rs<true, false>(a, chunk, blocks, smem, dev.device, st);
  if (a.out_bf16) return launch_rs<false, true>(a, chunk, blocks, smem, dev.device, st);
  return launch_rs<false, false>(a, chunk, blocks, smem, dev.device, st);
}
