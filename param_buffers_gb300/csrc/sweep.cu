// The memory-bound half of the step over the flat buffer: zero_, per-bucket gradient
// scaling, and the fused scale -> AdamW -> bf16 cast -> zero sweep (and its variant for
// a buffer of native MXFP8 parameters, which writes MX blocks instead of the bf16 cast).
//
// Pages: "05 · grad/param buffer: contiguous buffer data structures and read/write
// loop" (llm-infra-atlas) §6.3 (start_grad_sync multiplies each bucket by its
// gradient_scaling_factor), §6.5 (ZeRO-1 loop: the grad shard is read as fp32, Adam
// updates the fp32 master and m/v, the master is written back into param_data),
// §6.6 (zero_grad_buffer zeroes grad_data every iteration); "Megatron-LM architecture
// and source guide" (arganzheng.life) §6.4, steps 1-3 of DistributedOptimizer.step.
//
// Design: every kernel is a persistent grid-stride loop over 16-byte vectors (4 fp32
// elements), sized to 8 blocks of 256 threads per SM, with streaming (evict-first)
// loads and stores since every byte is touched exactly once.  The per-bucket factor
// comes from a segment table passed as a __grid_constant__ kernel parameter: the
// buckets plus the gaps between them, in offset order.  A thread's vector index only
// grows, so its segment cursor only moves forward (amortised O(1) lookup); a vector
// that straddles a segment boundary takes the per-element path.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <numeric>
#include <type_traits>
#include <vector>

#include "device.h"
#include "mx_block.cuh"
#include "sm100_ptx.cuh"

namespace {

using gtp::ptx::allow_dependents;
using gtp::ptx::wait_prior_grid;

constexpr int kThreads = 256;
constexpr int kBlocksPerSm = 8;
constexpr int kMaxBuckets = 512;

// Segment s covers elements [begin[s], begin[s+1]); begin[n] == numel.
template <int MAXS>
struct SegTable {
  int64_t begin[MAXS + 1];
  float factor[MAXS];
  int32_t active[MAXS];  // 1: a bucket; 0: a gap outside every bucket
  int32_t n;
};
constexpr int kSmallSegs = 2 * 32 + 1;
constexpr int kLargeSegs = 2 * kMaxBuckets + 1;
static_assert(sizeof(SegTable<kLargeSegs>) + 256 < 32764, "kernel parameter space");

template <int MAXS>
gtp_status build_segments(SegTable<MAXS> &t, int64_t numel, const gtp_bucket_desc *b,
                          const float *factors, int32_t nb) {
  std::vector<int32_t> ord(nb);
  std::iota(ord.begin(), ord.end(), 0);
  std::sort(ord.begin(), ord.end(), [&](int32_t x, int32_t y) { return b[x].offset < b[y].offset; });
  int n = 0;
  int64_t cur = 0;
  auto push = [&](int64_t beg, float f, int32_t act) {
    t.begin[n] = beg;
    t.factor[n] = f;
    t.active[n] = act;
    ++n;
  };
  for (int32_t k : ord) {
    const int64_t off = b[k].offset, len = b[k].numel;
    if (off < 0 || len < 0 || off > numel || len > numel - off)
      return gtp::fail(GTP_E_RANGE, "bucket %d [%lld, +%lld) outside [0, %lld)", k, (long long)off,
                       (long long)len, (long long)numel);
    if (len == 0) continue;
    if (off < cur)
      return gtp::fail(GTP_E_RANGE, "bucket %d at %lld overlaps the previous bucket (ends %lld)", k,
                       (long long)off, (long long)cur);
    if (off > cur) push(cur, 1.0f, 0);
    push(off, factors[k], 1);
    cur = off + len;
  }
  if (cur < numel || n == 0) push(cur, 1.0f, 0);
  t.begin[n] = numel;
  t.n = n;
  return GTP_OK;
}

struct AdamScalars {
  float decay;      // 1 - lr * wd
  float step_size;  // lr / (1 - b1^t)
  float sqrt_bc2;   // sqrt(1 - b2^t)
  float eps, b1, omb1, b2, omb2;
  int zero_grad;
  const float *grad_scale;  // device scalar (clip coefficient) or null
};

__device__ __forceinline__ void adam_update(float g, float &p, float &m, float &v,
                                            const AdamScalars &s) {
  m = fmaf(s.b1, m, s.omb1 * g);
  v = fmaf(s.b2, v, s.omb2 * (g * g));
  const float denom = sqrtf(v) / s.sqrt_bc2 + s.eps;
  p = p * s.decay - s.step_size * (m / denom);
}

template <int MAXS>
__device__ __forceinline__ int advance(const SegTable<MAXS> &t, int seg, int64_t e) {
  while (t.begin[seg + 1] <= e) ++seg;
  return seg;
}

// Four gradient elements of vector i as fp32 (the `.float()` of a bf16 gradient is exact),
// and their zeroing, for an fp32 or a bf16 grad buffer.
__device__ __forceinline__ float4 load_grad4(const float *g, int64_t i) {
  return __ldcs(reinterpret_cast<const float4 *>(g) + i);
}
__device__ __forceinline__ float4 load_grad4(const __nv_bfloat16 *g, int64_t i) {
  const uint2 w = __ldcs(reinterpret_cast<const uint2 *>(g) + i);
  const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162 *>(&w.x);
  const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162 *>(&w.y);
  return make_float4(__low2float(lo), __high2float(lo), __low2float(hi), __high2float(hi));
}
__device__ __forceinline__ void zero_grad4(float *g, int64_t i) {
  __stcs(reinterpret_cast<float4 *>(g) + i, make_float4(0.f, 0.f, 0.f, 0.f));
}
__device__ __forceinline__ void zero_grad4(__nv_bfloat16 *g, int64_t i) {
  __stcs(reinterpret_cast<uint2 *>(g) + i, make_uint2(0u, 0u));
}
__device__ __forceinline__ float grad_at(const float *g, int64_t e) { return g[e]; }
__device__ __forceinline__ float grad_at(const __nv_bfloat16 *g, int64_t e) { return __bfloat162float(g[e]); }
__device__ __forceinline__ void zero_at(float *g, int64_t e) { g[e] = 0.f; }
__device__ __forceinline__ void zero_at(__nv_bfloat16 *g, int64_t e) { g[e] = __float2bfloat16_rn(0.f); }

// GT: the grad buffer's element type, fp32 (grad_reduce_in_fp32) or bf16.
template <int MAXS, typename GT>
__global__ void __launch_bounds__(kThreads) adam_flat_kernel(
    GT *__restrict__ grad, float *__restrict__ master, float *__restrict__ exp_avg,
    float *__restrict__ exp_avg_sq, __nv_bfloat16 *__restrict__ param, int64_t numel,
    const AdamScalars s, const __grid_constant__ SegTable<MAXS> segs) {
  allow_dependents();
  wait_prior_grid();
  const bool clip = s.grad_scale != nullptr;
  const float cs = clip ? __ldg(s.grad_scale) : 1.f;
  const int64_t nvec = numel >> 2;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  int seg = 0;
  for (int64_t i = tid; i < nvec; i += stride) {
    const int64_t e0 = i << 2;
    float4 g4 = load_grad4(grad, i);
    float4 p4 = __ldcs(reinterpret_cast<const float4 *>(master) + i);
    float4 m4 = __ldcs(reinterpret_cast<const float4 *>(exp_avg) + i);
    float4 v4 = __ldcs(reinterpret_cast<const float4 *>(exp_avg_sq) + i);
    seg = advance(segs, seg, e0);
    float f0, f1, f2, f3;
    if (segs.begin[seg + 1] >= e0 + 4) {
      f0 = f1 = f2 = f3 = segs.factor[seg];
    } else {  // the vector straddles a bucket boundary
      f0 = segs.factor[seg];
      f1 = segs.factor[advance(segs, seg, e0 + 1)];
      f2 = segs.factor[advance(segs, seg, e0 + 2)];
      f3 = segs.factor[advance(segs, seg, e0 + 3)];
    }
    g4.x *= f0;  // the bucket scale, then the clip coefficient: two fp32 roundings, as in
    g4.y *= f1;  // an in-place scale of the buffer followed by an in-place clip
    g4.z *= f2;
    g4.w *= f3;
    if (clip) {
      g4.x *= cs; g4.y *= cs; g4.z *= cs; g4.w *= cs;
    }
    adam_update(g4.x, p4.x, m4.x, v4.x, s);
    adam_update(g4.y, p4.y, m4.y, v4.y, s);
    adam_update(g4.z, p4.z, m4.z, v4.z, s);
    adam_update(g4.w, p4.w, m4.w, v4.w, s);
    __stcs(reinterpret_cast<float4 *>(master) + i, p4);
    __stcs(reinterpret_cast<float4 *>(exp_avg) + i, m4);
    __stcs(reinterpret_cast<float4 *>(exp_avg_sq) + i, v4);
    const __nv_bfloat162 lo = __floats2bfloat162_rn(p4.x, p4.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(p4.z, p4.w);
    uint2 packed;
    packed.x = *reinterpret_cast<const uint32_t *>(&lo);
    packed.y = *reinterpret_cast<const uint32_t *>(&hi);
    __stcs(reinterpret_cast<uint2 *>(param) + i, packed);
    if (s.zero_grad) zero_grad4(grad, i);
  }
  // Ragged tail: numel % 4 elements, one per thread.
  const int64_t e = (nvec << 2) + tid;
  if (e < numel) {
    const int sg = advance(segs, 0, e);
    float p = master[e], m = exp_avg[e], v = exp_avg_sq[e];
    float g = grad_at(grad, e) * segs.factor[sg];
    if (clip) g *= cs;
    adam_update(g, p, m, v, s);
    master[e] = p;
    exp_avg[e] = m;
    exp_avg_sq[e] = v;
    param[e] = __float2bfloat16_rn(p);
    if (s.zero_grad) zero_at(grad, e);
  }
}

// The same sweep for a buffer of native MXFP8 parameters ("Generalized Tensor Parallelism
// (GTP)" §1.3: the optimizer writes the FP8 weight from the fp32 master once per step):
// instead of a bf16 copy, every aligned 32-element block of the updated master becomes 32
// E4M3 codes in param_data (uint8, the buffer's storage dtype) and one E8M0 scale byte.
// A parameter view [N, K] starting at a multiple of 32 with K % 32 == 0 is then exactly
// the rowwise MXFP8 view the forward GEMM consumes.  Eight neighbouring lanes hold one
// block (lane i owns elements 4i..4i+3 of a warp's 128), so the block's amax and its
// finite flag take three butterfly shuffles; the loop runs warp-uniformly so every lane
// reaches the shuffles.  numel is a multiple of 32, so a block is never split.
template <int MAXS>
__global__ void __launch_bounds__(kThreads) adam_flat_mx_kernel(
    float *__restrict__ grad, float *__restrict__ master, float *__restrict__ exp_avg,
    float *__restrict__ exp_avg_sq, uint8_t *__restrict__ e4m3, uint8_t *__restrict__ e8m0, int64_t numel,
    const AdamScalars s, const __grid_constant__ SegTable<MAXS> segs) {
  allow_dependents();
  wait_prior_grid();
  const bool clip = s.grad_scale != nullptr;
  const float cs = clip ? __ldg(s.grad_scale) : 1.f;
  const int lane = threadIdx.x & 31;
  const int64_t nvec = numel >> 2;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const int64_t warp0 = int64_t(blockIdx.x) * blockDim.x + (threadIdx.x & ~31);
  int seg = 0;
  for (int64_t base = warp0; base < nvec; base += stride) {
    const int64_t i = base + lane;
    const bool valid = i < nvec;  // whole 8-lane groups agree: nvec % 8 == 0
    float4 p4 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (valid) {
      const int64_t e0 = i << 2;
      float4 g4 = __ldcs(reinterpret_cast<const float4 *>(grad) + i);
      p4 = __ldcs(reinterpret_cast<const float4 *>(master) + i);
      float4 m4 = __ldcs(reinterpret_cast<const float4 *>(exp_avg) + i);
      float4 v4 = __ldcs(reinterpret_cast<const float4 *>(exp_avg_sq) + i);
      seg = advance(segs, seg, e0);
      float f0, f1, f2, f3;
      if (segs.begin[seg + 1] >= e0 + 4) {
        f0 = f1 = f2 = f3 = segs.factor[seg];
      } else {
        f0 = segs.factor[seg];
        f1 = segs.factor[advance(segs, seg, e0 + 1)];
        f2 = segs.factor[advance(segs, seg, e0 + 2)];
        f3 = segs.factor[advance(segs, seg, e0 + 3)];
      }
      g4.x *= f0;
      g4.y *= f1;
      g4.z *= f2;
      g4.w *= f3;
      if (clip) {
        g4.x *= cs; g4.y *= cs; g4.z *= cs; g4.w *= cs;
      }
      adam_update(g4.x, p4.x, m4.x, v4.x, s);
      adam_update(g4.y, p4.y, m4.y, v4.y, s);
      adam_update(g4.z, p4.z, m4.z, v4.z, s);
      adam_update(g4.w, p4.w, m4.w, v4.w, s);
      __stcs(reinterpret_cast<float4 *>(master) + i, p4);
      __stcs(reinterpret_cast<float4 *>(exp_avg) + i, m4);
      __stcs(reinterpret_cast<float4 *>(exp_avg_sq) + i, v4);
      if (s.zero_grad) __stcs(reinterpret_cast<float4 *>(grad) + i, make_float4(0.f, 0.f, 0.f, 0.f));
    }
    float amax = fmaxf(fmaxf(fabsf(p4.x), fabsf(p4.y)), fmaxf(fabsf(p4.z), fabsf(p4.w)));
    int fin = (isfinite(p4.x) && isfinite(p4.y) && isfinite(p4.z) && isfinite(p4.w)) ? 1 : 0;
#pragma unroll
    for (int d = 1; d < 8; d <<= 1) {
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, d));
      fin &= __shfl_xor_sync(0xFFFFFFFFu, fin, d);
    }
    uint32_t sbyte, codes;
    if (fin) {
      sbyte = gtp::mx::scale_byte(amax);
      const float inv = gtp::mx::inv_scale(sbyte);
      codes = gtp::mx::encode4(p4.x * inv, p4.y * inv, p4.z * inv, p4.w * inv);
    } else {
      sbyte = gtp::mx::kNanScale;
      codes = gtp::mx::kNanCodes;
    }
    // the warp's four scale bytes (lanes 0, 8, 16, 24) leave as one 4-byte word
    const uint32_t word = __shfl_sync(0xFFFFFFFFu, sbyte, 0) | (__shfl_sync(0xFFFFFFFFu, sbyte, 8) << 8) |
                          (__shfl_sync(0xFFFFFFFFu, sbyte, 16) << 16) | (__shfl_sync(0xFFFFFFFFu, sbyte, 24) << 24);
    if (valid) {
      __stcs(reinterpret_cast<uint32_t *>(e4m3) + i, codes);
      if (lane == 0) {
        if (base + 32 <= nvec)
          __stcs(reinterpret_cast<uint32_t *>(e8m0) + (base >> 5), word);
        else  // the last, partial warp of the buffer: only its whole blocks
          for (int b = 0; b < int((nvec - base) >> 3); ++b) e8m0[(base >> 3) + b] = uint8_t(word >> (8 * b));
      }
    }
  }
}

template <int MAXS>
__global__ void __launch_bounds__(kThreads) bucket_scale_kernel(float *__restrict__ grad, int64_t numel,
                                                                const __grid_constant__ SegTable<MAXS> segs) {
  allow_dependents();
  wait_prior_grid();
  const int64_t nvec = numel >> 2;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  int seg = 0;
  for (int64_t i = tid; i < nvec; i += stride) {
    const int64_t e0 = i << 2;
    seg = advance(segs, seg, e0);
    if (segs.begin[seg + 1] >= e0 + 4) {
      if (!segs.active[seg]) continue;  // a gap between buckets: not touched
      const float f = segs.factor[seg];
      float4 g = __ldcs(reinterpret_cast<const float4 *>(grad) + i);
      g.x *= f; g.y *= f; g.z *= f; g.w *= f;
      __stcs(reinterpret_cast<float4 *>(grad) + i, g);
    } else {
      for (int j = 0; j < 4; ++j) {
        const int sg = advance(segs, seg, e0 + j);
        if (segs.active[sg]) grad[e0 + j] *= segs.factor[sg];
      }
    }
  }
  const int64_t e = (nvec << 2) + tid;
  if (e < numel) {
    const int sg = advance(segs, 0, e);
    if (segs.active[sg]) grad[e] *= segs.factor[sg];
  }
}

__global__ void __launch_bounds__(kThreads) zero_kernel(uint8_t *__restrict__ data, int64_t nbytes) {
  allow_dependents();
  wait_prior_grid();
  const int64_t nvec = nbytes >> 4;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  for (int64_t i = tid; i < nvec; i += stride)
    __stcs(reinterpret_cast<uint4 *>(data) + i, make_uint4(0u, 0u, 0u, 0u));
  const int64_t b = (nvec << 4) + tid;
  if (b < nbytes) data[b] = 0;
}

int grid_for(int64_t nvec, int sm_count) {
  const int64_t want = (nvec + kThreads - 1) / kThreads;
  return int(std::max<int64_t>(1, std::min<int64_t>(want, int64_t(sm_count) * kBlocksPerSm)));
}

gtp_status check_buckets_args(const gtp_bucket_desc *buckets, const float *factors, int32_t nb) {
  if (nb < 0) return gtp::fail(GTP_E_ARG, "n_buckets < 0");
  if (nb > kMaxBuckets) return gtp::fail(GTP_E_CAPACITY, "%d buckets > %d supported", nb, kMaxBuckets);
  if (nb > 0 && (!buckets || !factors)) return gtp::fail(GTP_E_ARG, "null buckets or factors");
  return GTP_OK;
}

}  // namespace

namespace gtp {
// Zeroes `nbytes` bytes at a 16-byte-aligned device pointer (the degenerate GEMM cases
// whose output is all zeros use it).
gtp_status launch_zero_bytes(void *data, int64_t nbytes, cudaStream_t stream, int sm_count) {
  if (nbytes <= 0) return GTP_OK;
  return launch_overlapped(zero_kernel, grid_for(nbytes >> 4, sm_count), kThreads, 0, stream, "zero",
                           static_cast<uint8_t *>(data), nbytes);
}
}  // namespace gtp

extern "C" gtp_status gtp_buffer_zero(void *data, gtp_dtype dt, int64_t numel, gtp_stream stream) {
  gtp::clear_error();
  int64_t es = 0;
  switch (dt) {
    case GTP_F32: es = 4; break;
    case GTP_BF16: case GTP_F16: es = 2; break;
    case GTP_U8: es = 1; break;
    default: return gtp::fail(GTP_E_DTYPE, "dtype %d", int(dt));
  }
  if (numel < 0) return gtp::fail(GTP_E_ARG, "numel < 0");
  if (numel == 0) return GTP_OK;
  if (!data) return gtp::fail(GTP_E_ARG, "null data");
  if (!gtp::aligned16(data)) return gtp::fail(GTP_E_ALIGN, "data not 16-byte aligned");
  gtp::DeviceInfo dev;
  if (gtp_status st = gtp::require_sm103(&dev)) return st;
  const int64_t nbytes = numel * es;
  return gtp::launch_overlapped(zero_kernel, grid_for(nbytes >> 4, dev.sm_count), kThreads, 0, gtp::as_stream(stream),
                                "buffer_zero", static_cast<uint8_t *>(data), nbytes);
}

extern "C" gtp_status gtp_bucket_scale(float *grad_data, int64_t grad_numel, const gtp_bucket_desc *buckets,
                                       const float *factors, int32_t n_buckets, gtp_stream stream) {
  gtp::clear_error();
  if (gtp_status st = check_buckets_args(buckets, factors, n_buckets)) return st;
  if (grad_numel < 0) return gtp::fail(GTP_E_ARG, "grad_numel < 0");
  if (grad_numel > 0 && !grad_data) return gtp::fail(GTP_E_ARG, "null grad_data");
  if (grad_numel > 0 && !gtp::aligned16(grad_data)) return gtp::fail(GTP_E_ALIGN, "grad_data not 16-byte aligned");
  const int64_t nvec = grad_numel >> 2;
  if (n_buckets <= 32) {
    SegTable<kSmallSegs> t;
    if (gtp_status st = build_segments(t, grad_numel, buckets, factors, n_buckets)) return st;
    if (grad_numel == 0) return GTP_OK;
    gtp::DeviceInfo dev;
    if (gtp_status st = gtp::require_sm103(&dev)) return st;
    return gtp::launch_overlapped(bucket_scale_kernel<kSmallSegs>, grid_for(nvec, dev.sm_count), kThreads, 0,
                                  gtp::as_stream(stream), "bucket_scale", grad_data, grad_numel, t);
  } else {
    SegTable<kLargeSegs> t;
    if (gtp_status st = build_segments(t, grad_numel, buckets, factors, n_buckets)) return st;
    if (grad_numel == 0) return GTP_OK;
    gtp::DeviceInfo dev;
    if (gtp_status st = gtp::require_sm103(&dev)) return st;
    return gtp::launch_overlapped(bucket_scale_kernel<kLargeSegs>, grid_for(nvec, dev.sm_count), kThreads, 0,
                                  gtp::as_stream(stream), "bucket_scale", grad_data, grad_numel, t);
  }
  return gtp::check_launch("bucket_scale");
}

namespace {

// Validates the hyper-parameters and the shared buffers and folds the step's constants.
gtp_status adam_prologue(const float *grad_data, const float *master, const float *exp_avg, const float *exp_avg_sq,
                         int64_t numel, const gtp_bucket_desc *buckets, const float *factors, int32_t n_buckets,
                         const gtp_adam_hparams *h, AdamScalars &s) {
  if (!h) return gtp::fail(GTP_E_ARG, "null hparams");
  if (gtp_status st = check_buckets_args(buckets, factors, n_buckets)) return st;
  if (numel < 0) return gtp::fail(GTP_E_ARG, "numel < 0");
  if (!(h->lr >= 0.f) || !(h->beta1 >= 0.f && h->beta1 < 1.f) || !(h->beta2 >= 0.f && h->beta2 < 1.f) ||
      !(h->eps >= 0.f) || !(h->weight_decay >= 0.f) || h->step < 1 ||
      (h->zero_grad_after != 0 && h->zero_grad_after != 1))
    return gtp::fail(GTP_E_ARG, "hyper-parameters out of range (lr, wd, eps >= 0; 0 <= beta < 1; step >= 1)");
  if (numel > 0) {
    if (!grad_data || !master || !exp_avg || !exp_avg_sq) return gtp::fail(GTP_E_ARG, "null buffer pointer");
    if (!gtp::aligned16(grad_data) || !gtp::aligned16(master) || !gtp::aligned16(exp_avg) ||
        !gtp::aligned16(exp_avg_sq))
      return gtp::fail(GTP_E_ALIGN, "buffer pointers must be 16-byte aligned");
  }
  const double t = double(h->step);
  const double bc1 = 1.0 - std::pow(double(h->beta1), t);
  const double bc2 = 1.0 - std::pow(double(h->beta2), t);
  if (!(bc1 > 0.0) || !(bc2 > 0.0)) return gtp::fail(GTP_E_ARG, "bias correction underflows to 0");
  s.decay = float(1.0 - double(h->lr) * double(h->weight_decay));
  s.step_size = float(double(h->lr) / bc1);
  s.sqrt_bc2 = float(std::sqrt(bc2));
  s.eps = h->eps;
  s.b1 = h->beta1;
  s.omb1 = float(1.0 - double(h->beta1));
  s.b2 = h->beta2;
  s.omb2 = float(1.0 - double(h->beta2));
  s.zero_grad = h->zero_grad_after;
  s.grad_scale = h->grad_scale;
  if (reinterpret_cast<uintptr_t>(s.grad_scale) & 3u)
    return gtp::fail(GTP_E_ALIGN, "grad_scale must be 4-byte aligned");
  return GTP_OK;
}

// The sweep updates its arrays element by element in place, so no two may share a byte:
// an overlap would read bytes that another array's store of the same pass has changed.
struct Span {
  const void *p;
  int64_t bytes;
  const char *name;
};
gtp_status check_distinct(const Span *a, int n) {
  for (int i = 0; i < n; ++i)
    for (int j = i + 1; j < n; ++j) {
      const uintptr_t lo_i = reinterpret_cast<uintptr_t>(a[i].p), lo_j = reinterpret_cast<uintptr_t>(a[j].p);
      if (a[i].bytes > 0 && a[j].bytes > 0 && lo_i < lo_j + uintptr_t(a[j].bytes) && lo_j < lo_i + uintptr_t(a[i].bytes))
        return gtp::fail(GTP_E_ARG, "%s overlaps %s", a[i].name, a[j].name);
    }
  return GTP_OK;
}

// Builds the segment table that fits n_buckets and launches kernel<table size>.
template <typename Launch>
gtp_status with_segments(int64_t numel, const gtp_bucket_desc *buckets, const float *factors, int32_t n_buckets,
                         Launch &&launch) {
  auto run = [&](auto &tab) -> gtp_status {
    if (gtp_status st = build_segments(tab, numel, buckets, factors, n_buckets)) return st;
    if (numel == 0) return GTP_OK;
    gtp::DeviceInfo dev;
    if (gtp_status st = gtp::require_sm103(&dev)) return st;
    return launch(tab, grid_for(numel >> 2, dev.sm_count));
  };
  if (n_buckets <= 32) {
    SegTable<kSmallSegs> tab;
    return run(tab);
  }
  SegTable<kLargeSegs> tab;
  return run(tab);
}

template <typename T>
struct SegSize;
template <int MAXS>
struct SegSize<SegTable<MAXS>> {
  static constexpr int value = MAXS;
};

}  // namespace

extern "C" gtp_status gtp_adam_step_flat(float *grad_data, float *master, float *exp_avg, float *exp_avg_sq,
                                         void *param_data, int64_t numel, const gtp_bucket_desc *buckets,
                                         const float *factors, int32_t n_buckets, const gtp_adam_hparams *h,
                                         gtp_stream stream) {
  gtp::clear_error();
  AdamScalars s;
  if (gtp_status st = adam_prologue(grad_data, master, exp_avg, exp_avg_sq, numel, buckets, factors, n_buckets, h, s))
    return st;
  if (numel > 0 && !param_data) return gtp::fail(GTP_E_ARG, "null buffer pointer");
  if (numel > 0 && !gtp::aligned16(param_data)) return gtp::fail(GTP_E_ALIGN, "buffer pointers must be 16-byte aligned");
  const Span arrays[5] = {{grad_data, 4 * numel, "grad_data"}, {master, 4 * numel, "master"},
                          {exp_avg, 4 * numel, "exp_avg"}, {exp_avg_sq, 4 * numel, "exp_avg_sq"},
                          {param_data, 2 * numel, "param_data"}};
  if (gtp_status st = check_distinct(arrays, 5)) return st;
  auto *param = static_cast<__nv_bfloat16 *>(param_data);
  return with_segments(numel, buckets, factors, n_buckets, [&](auto &tab, int grid) {
    constexpr int S = SegSize<std::decay_t<decltype(tab)>>::value;
    return gtp::launch_overlapped(adam_flat_kernel<S, float>, grid, kThreads, 0, gtp::as_stream(stream),
                                  "adam_step_flat", grad_data, master, exp_avg, exp_avg_sq, param, numel, s, tab);
  });
}

extern "C" gtp_status gtp_adam_step_flat_bf16_grad(void *grad_data, float *master, float *exp_avg, float *exp_avg_sq,
                                                   void *param_data, int64_t numel, const gtp_bucket_desc *buckets,
                                                   const float *factors, int32_t n_buckets, const gtp_adam_hparams *h,
                                                   gtp_stream stream) {
  gtp::clear_error();
  AdamScalars s;
  if (gtp_status st = adam_prologue(static_cast<const float *>(grad_data), master, exp_avg, exp_avg_sq, numel, buckets,
                                    factors, n_buckets, h, s))
    return st;
  if (numel > 0 && !param_data) return gtp::fail(GTP_E_ARG, "null buffer pointer");
  if (numel > 0 && !gtp::aligned16(param_data)) return gtp::fail(GTP_E_ALIGN, "buffer pointers must be 16-byte aligned");
  const Span arrays[5] = {{grad_data, 2 * numel, "grad_data"}, {master, 4 * numel, "master"},
                          {exp_avg, 4 * numel, "exp_avg"}, {exp_avg_sq, 4 * numel, "exp_avg_sq"},
                          {param_data, 2 * numel, "param_data"}};
  if (gtp_status st = check_distinct(arrays, 5)) return st;
  auto *grad = static_cast<__nv_bfloat16 *>(grad_data);
  auto *param = static_cast<__nv_bfloat16 *>(param_data);
  return with_segments(numel, buckets, factors, n_buckets, [&](auto &tab, int grid) {
    constexpr int S = SegSize<std::decay_t<decltype(tab)>>::value;
    return gtp::launch_overlapped(adam_flat_kernel<S, __nv_bfloat16>, grid, kThreads, 0, gtp::as_stream(stream),
                                  "adam_step_flat_bf16_grad", grad, master, exp_avg, exp_avg_sq, param, numel, s, tab);
  });
}

extern "C" gtp_status gtp_adam_step_flat_mxfp8(float *grad_data, float *master, float *exp_avg, float *exp_avg_sq,
                                               uint8_t *param_e4m3, uint8_t *param_e8m0, int64_t numel,
                                               const gtp_bucket_desc *buckets, const float *factors,
                                               int32_t n_buckets, const gtp_adam_hparams *h, gtp_stream stream) {
  gtp::clear_error();
  AdamScalars s;
  if (gtp_status st = adam_prologue(grad_data, master, exp_avg, exp_avg_sq, numel, buckets, factors, n_buckets, h, s))
    return st;
  if (numel % 32) return gtp::fail(GTP_E_SHAPE, "numel must be a multiple of 32 (whole MX blocks)");
  if (numel > 0 && (!param_e4m3 || !param_e8m0)) return gtp::fail(GTP_E_ARG, "null param_e4m3 or param_e8m0");
  if (numel > 0 && !gtp::aligned16(param_e4m3)) return gtp::fail(GTP_E_ALIGN, "param_e4m3 must be 16-byte aligned");
  if (numel > 0 && (reinterpret_cast<uintptr_t>(param_e8m0) & 3u))
    return gtp::fail(GTP_E_ALIGN, "param_e8m0 must be 4-byte aligned");
  const Span arrays[6] = {{grad_data, 4 * numel, "grad_data"}, {master, 4 * numel, "master"},
                          {exp_avg, 4 * numel, "exp_avg"},     {exp_avg_sq, 4 * numel, "exp_avg_sq"},
                          {param_e4m3, numel, "param_e4m3"},  {param_e8m0, numel / 32, "param_e8m0"}};
  if (gtp_status st = check_distinct(arrays, 6)) return st;
  return with_segments(numel, buckets, factors, n_buckets, [&](auto &tab, int grid) {
    constexpr int S = SegSize<std::decay_t<decltype(tab)>>::value;
    return gtp::launch_overlapped(adam_flat_mx_kernel<S>, grid, kThreads, 0, gtp::as_stream(stream),
                                  "adam_step_flat_mxfp8", grad_data, master, exp_avg, exp_avg_sq, param_e4m3,
                                  param_e8m0, numel, s, tab);
  });
}
