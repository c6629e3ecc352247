// Per-bucket gradient norms, a non-finite check and the global-norm clip coefficient.
//
// Pages: "05 · grad/param buffer: contiguous buffer data structures and read/write loop"
// (llm-infra-atlas) §6.3: with check_for_nan_in_grad / check_for_large_grads,
// start_grad_sync computes the L2 norm of each bucket's grad_data before the collective
// (NaN/Inf fatal, abnormally large non-fatal); "Megatron-LM architecture and source
// guide" (arganzheng.life) §4: --clip-grad 1.0, and optimizer.step() returns grad_norm.
// Reading: the norm is taken of the scaled gradient (factor_b * g, the value the
// optimizer consumes), and clipping follows the usual global-norm rule
// coef = min(1, max_norm / (norm + 1e-6)); the optimizer sweep multiplies by coef.
//
// Two launches, deterministic (no atomics, fixed reduction order):
//   1. one block per 64K-element chunk of one bucket: fp32 sums of squares in four
//      interleaved accumulators per thread, combined in fp64, block-reduced in fp64; one
//      (sum, non-finite count) partial per chunk into the workspace;
//   2. one block (1024 threads, or 128 for up to 4096 partials: fp64 arithmetic is slow on
//      this part and every thread of the block takes part in the reductions): each
//      bucket's partials summed in a fixed tree, then the total norm and the clip
//      coefficient.
// HBM-bound: 4 bytes read per element.
#include <cmath>
#include <mutex>
#include <vector>

#include "device.h"
#include "sm100_ptx.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int64_t kChunk = 65536;  // elements reduced by one block
constexpr int kMaxBuckets = 512;
constexpr int kFinThreads = 1024;  // the finalize block at most; 128 for up to 4096 partials
constexpr int kFinThreadsSmall = 128;

struct Partial {
  double sumsq;
  uint32_t nonfinite;
  uint32_t pad;
};
static_assert(sizeof(Partial) == 16, "partial layout");

struct NormTable {
  int64_t offset[kMaxBuckets];
  int64_t numel[kMaxBuckets];
  float factor[kMaxBuckets];
  int32_t chunk_begin[kMaxBuckets + 1];  // prefix sums of chunks per bucket
  int32_t n;
};
static_assert(sizeof(NormTable) + 256 < 32764, "kernel parameter space");

__device__ __forceinline__ int bucket_of_chunk(const NormTable &t, int c) {
  int lo = 0, hi = t.n - 1;  // largest b with chunk_begin[b] <= c
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (t.chunk_begin[mid] <= c) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ double block_sum_f64(double v, double *red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  double s = 0.0;  // the warps' sums, reduced by warp 0 in the same butterfly order
  if (w == 0) {
    s = l < int(blockDim.x >> 5) ? red[l] : 0.0;
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
  }
  return s;  // valid in thread 0
}

__device__ __forceinline__ uint32_t block_sum_u32(uint32_t v, uint32_t *red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  uint32_t s = 0;
  if (threadIdx.x == 0)
    for (int i = 0; i < int(blockDim.x >> 5); ++i) s += red[i];
  return s;
}

__global__ void __launch_bounds__(kThreads) grad_norm_partials_kernel(const float *__restrict__ grad,
                                                                      Partial *__restrict__ partials,
                                                                      const __grid_constant__ NormTable t) {
  __shared__ double red_d[kThreads / 32];
  __shared__ uint32_t red_u[kThreads / 32];
  gtp::ptx::allow_dependents();
  gtp::ptx::wait_prior_grid();
  const int c = blockIdx.x;
  const int b = bucket_of_chunk(t, c);
  const int64_t lo = t.offset[b] + int64_t(c - t.chunk_begin[b]) * kChunk;
  const int64_t hi = min(lo + kChunk, t.offset[b] + t.numel[b]);
  const float f = t.factor[b];
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  uint32_t bad = 0;
  // scalar head up to a 16-byte boundary, float4 body, scalar tail
  const int64_t body0 = min(hi, (lo + 3) & ~int64_t(3));
  const int64_t body1 = max(body0, hi & ~int64_t(3));
  for (int64_t i = lo + threadIdx.x; i < body0; i += blockDim.x) {
    const float v = grad[i] * f;
    bad += isfinite(v) ? 0u : 1u;
    acc[0] = fmaf(v, v, acc[0]);
  }
  for (int64_t i = (body0 >> 2) + threadIdx.x; i < (body1 >> 2); i += blockDim.x) {
    const float4 g = __ldcs(reinterpret_cast<const float4 *>(grad) + i);
    const float v0 = g.x * f, v1 = g.y * f, v2 = g.z * f, v3 = g.w * f;
    bad += (isfinite(v0) ? 0u : 1u) + (isfinite(v1) ? 0u : 1u) + (isfinite(v2) ? 0u : 1u) + (isfinite(v3) ? 0u : 1u);
    acc[0] = fmaf(v0, v0, acc[0]);
    acc[1] = fmaf(v1, v1, acc[1]);
    acc[2] = fmaf(v2, v2, acc[2]);
    acc[3] = fmaf(v3, v3, acc[3]);
  }
  for (int64_t i = body1 + threadIdx.x; i < hi; i += blockDim.x) {
    const float v = grad[i] * f;
    bad += isfinite(v) ? 0u : 1u;
    acc[1] = fmaf(v, v, acc[1]);
  }
  const double mine = (double(acc[0]) + double(acc[1])) + (double(acc[2]) + double(acc[3]));
  const double s = block_sum_f64(mine, red_d);
  const uint32_t n = block_sum_u32(bad, red_u);
  if (threadIdx.x == 0) partials[c] = Partial{s, n, 0u};
}

__global__ void __launch_bounds__(kFinThreads) grad_norm_finalize_kernel(
    const Partial *__restrict__ partials, double *__restrict__ sumsq, uint32_t *__restrict__ nonfinite,
    float *__restrict__ total_norm, float *__restrict__ clip_coef, float max_norm, const __grid_constant__ NormTable t) {
  __shared__ double red_d[kFinThreads / 32];
  __shared__ uint32_t red_u[kFinThreads / 32];
  gtp::ptx::allow_dependents();
  gtp::ptx::wait_prior_grid();
  double total = 0.0;
  for (int b = 0; b < t.n; ++b) {
    double s = 0.0;
    uint32_t n = 0;
    for (int c = t.chunk_begin[b] + threadIdx.x; c < t.chunk_begin[b + 1]; c += blockDim.x) {
      s += partials[c].sumsq;
      n += partials[c].nonfinite;
    }
    s = block_sum_f64(s, red_d);
    n = block_sum_u32(n, red_u);
    if (threadIdx.x == 0) {
      sumsq[b] = s;
      nonfinite[b] = n;
      total += s;
    }
  }
  if (threadIdx.x == 0) {
    const double norm = sqrt(total);
    *total_norm = float(norm);
    double coef = 1.0;
    if (max_norm > 0.f) coef = fmin(1.0, double(max_norm) / (norm + 1e-6));
    *clip_coef = float(coef);
  }
}

gtp_status build_table(NormTable &t, int64_t numel, const gtp_bucket_desc *b, const float *factors, int32_t nb,
                       int64_t *n_chunks) {
  if (nb < 1) return gtp::fail(GTP_E_ARG, "at least one bucket is required");
  if (nb > kMaxBuckets) return gtp::fail(GTP_E_CAPACITY, "%d buckets > %d supported", nb, kMaxBuckets);
  if (!b || !factors) return gtp::fail(GTP_E_ARG, "null buckets or factors");
  int64_t chunks = 0;
  t.n = nb;
  for (int32_t k = 0; k < nb; ++k) {
    const int64_t off = b[k].offset, len = b[k].numel;
    if (off < 0 || len < 0 || off > numel || len > numel - off)
      return gtp::fail(GTP_E_RANGE, "bucket %d [%lld, +%lld) outside [0, %lld)", k, (long long)off, (long long)len,
                       (long long)numel);
    t.offset[k] = off;
    t.numel[k] = len;
    t.factor[k] = factors[k];
    t.chunk_begin[k] = int32_t(chunks);
    chunks += (len + kChunk - 1) / kChunk;
    if (chunks > (int64_t(1) << 30)) return gtp::fail(GTP_E_SHAPE, "too many elements");
  }
  t.chunk_begin[nb] = int32_t(chunks);
  *n_chunks = chunks;
  return GTP_OK;
}

}  // namespace

namespace gtp {

// Shared by the allocating and the non-allocating entry points: validates, then launches
// both kernels with `workspace` holding the chunk partials.
gtp_status grad_norm_run(const float *grad_data, int64_t numel, const gtp_bucket_desc *buckets, const float *factors,
                         int32_t n_buckets, float max_norm, void *workspace, size_t workspace_bytes, double *sumsq,
                         uint32_t *nonfinite, float *total_norm, float *clip_coef, gtp_stream stream) {
  if (numel < 0) return fail(GTP_E_ARG, "numel < 0");
  if (!(max_norm >= 0.f)) return fail(GTP_E_ARG, "max_norm must be >= 0 (0 disables clipping)");
  NormTable t;
  int64_t chunks = 0;
  if (gtp_status s = build_table(t, numel, buckets, factors, n_buckets, &chunks)) return s;
  if (!sumsq || !nonfinite || !total_norm || !clip_coef) return fail(GTP_E_ARG, "null output pointer");
  if (numel > 0 && !grad_data) return fail(GTP_E_ARG, "null grad_data");
  if (numel > 0 && !aligned16(grad_data)) return fail(GTP_E_ALIGN, "grad_data must be 16-byte aligned");
  const size_t need = size_t(chunks) * sizeof(Partial);
  if (chunks > 0 && (!workspace || workspace_bytes < need))
    return fail(GTP_E_CAPACITY, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
  if (chunks > 0 && (reinterpret_cast<uintptr_t>(workspace) & 15u)) return fail(GTP_E_ALIGN, "workspace alignment");
  DeviceInfo dev;
  if (gtp_status s = require_sm103(&dev)) return s;
  cudaStream_t st = as_stream(stream);
  Partial *partials = static_cast<Partial *>(workspace);
  if (chunks > 0)
    if (gtp_status s = launch_overlapped(grad_norm_partials_kernel, dim3(unsigned(chunks)), kThreads, 0, st,
                                         "grad_norm_partials", grad_data, partials, t))
      return s;
  // A small input's few partials go to a small block: every thread of the block takes part
  // in the fp64 reductions, and fp64 arithmetic is slow on this part.
  const int fin_threads = chunks > 4096 ? kFinThreads : kFinThreadsSmall;
  return launch_overlapped(grad_norm_finalize_kernel, 1, fin_threads, 0, st, "grad_norm_finalize",
                           const_cast<const Partial *>(partials), sumsq, nonfinite, total_norm, clip_coef, max_norm, t);
}

}  // namespace gtp

extern "C" size_t gtp_grad_norm_workspace_bytes(const gtp_bucket_desc *buckets, int32_t n_buckets) {
  if (!buckets || n_buckets < 0) return 0;
  size_t chunks = 0;
  for (int32_t k = 0; k < n_buckets; ++k)
    if (buckets[k].numel > 0) chunks += size_t((buckets[k].numel + kChunk - 1) / kChunk);
  return chunks * sizeof(Partial);
}

extern "C" gtp_status gtp_grad_norm(const float *grad_data, int64_t numel, const gtp_bucket_desc *buckets,
                                    const float *factors, int32_t n_buckets, float max_norm, void *workspace,
                                    size_t workspace_bytes, double *sumsq, uint32_t *nonfinite, float *total_norm,
                                    float *clip_coef, gtp_stream stream) {
  gtp::clear_error();
  return gtp::grad_norm_run(grad_data, numel, buckets, factors, n_buckets, max_norm, workspace, workspace_bytes, sumsq,
                            nonfinite, total_norm, clip_coef, stream);
}

// ------------------------------------------------------------------ non-allocating variant
//
// Some callers cannot allocate device memory at the point where they need the gradient
// norm: code running under a fixed memory budget whose allocator must not be re-entered
// (a caching allocator's out-of-memory handler, a custom arena that is already full), or
// a plain C caller without an allocator of its own that still wants a result.  For them
// gtp_grad_norm_noalloc keeps its per-chunk partials in the array below instead of a
// caller workspace.  The array lives in the library's device image, so every GPU that
// loads the library holds its 1 MiB until the process exits.
namespace {
constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 65536 chunk partials
static __device__ __align__(256) uint8_t g_norm_scratch[kNoAllocScratchBytes];

constexpr int kMaxScratchDevices = 64;
void *g_scratch_ptr[kMaxScratchDevices];  // written under g_scratch_mutex, only ever once a lookup succeeds
std::mutex g_scratch_mutex;

// The device address of the scratch array on the current device `dev`.  Only a successful
// lookup is kept: a lookup that fails (a sticky error from earlier work, say) is retried by
// the next call instead of failing every later call on that device.
cudaError_t scratch_address(int dev, void **out) {
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_norm_scratch);
    if (e != cudaSuccess) return e;
    if (!p) return cudaErrorInvalidSymbol;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}
}  // namespace

extern "C" gtp_status gtp_grad_norm_noalloc(const float *grad_data, int64_t numel, const gtp_bucket_desc *buckets,
                                            const float *factors, int32_t n_buckets, float max_norm, double *sumsq,
                                            uint32_t *nonfinite, float *total_norm, float *clip_coef,
                                            gtp_stream stream) {
  gtp::clear_error();
  if (n_buckets > 0 && buckets) {
    const size_t need = gtp_grad_norm_workspace_bytes(buckets, n_buckets);
    if (need > kNoAllocScratchBytes)
      return gtp::fail(GTP_E_CAPACITY,
                       "gtp_grad_norm_noalloc: %zu bytes of partials needed, its fixed scratch holds %zu "
                       "(at most 65536 chunks of 65536 elements); use gtp_grad_norm with a workspace",
                       need, kNoAllocScratchBytes);
  }
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return gtp::fail(GTP_E_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxScratchDevices) return gtp::fail(GTP_E_DEVICE, "device ordinal %d unsupported", dev);
  // First call on this device: resolve the device address of the scratch array (the
  // host-side name is only a stand-in), with this device current.
  void *scratch = nullptr;
  e = scratch_address(dev, &scratch);
  if (e != cudaSuccess) return gtp::fail(GTP_E_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
  return gtp::grad_norm_run(grad_data, numel, buckets, factors, n_buckets, max_norm, scratch, kNoAllocScratchBytes,
                            sumsq, nonfinite, total_norm, clip_coef, stream);
}
