// The three GEMMs of one tensor-parallel linear shard on the 5th-generation tensor cores.
//
// Page: "01 · ColumnParallelLinear / RowParallelLinear and the core autograd"
// (llm-infra-atlas), §4.1 (forward: output = total_input · weight^T) and §4.2 (backward:
// dgrad = grad_output · weight; wgrad with gradient_accumulation_fusion accumulated in
// fp32 straight into weight.main_grad), with main_grad a view of the flat grad buffer
// ("05 · grad/param buffer ...", §5).
//
// One persistent, warp-specialised kernel serves all three products D (+)= A · B^T:
//   warp 0      TMA producer: 128x64 A and 256x64 B bf16 tiles, 128-byte swizzle, into
//               a 4-stage shared-memory ring (mbarrier full/empty pairs);
//   warp 1      allocates 512 tensor-memory columns (two 128x256 fp32 accumulators) and
//               issues tcgen05.mma (M=128, N=256, K=16) from one thread;
//   warps 2-5   epilogue: tcgen05.ld of their 32-lane quarter, staged through swizzled
//               shared memory, written by TMA - a bf16 store (fprop, dgrad) or an fp32
//               reduce-add into main_grad (wgrad).  The accumulator is double-buffered,
//               so the epilogue of one tile overlaps the main loop of the next.
// Operand majorness comes from the descriptors, never from a transpose in memory:
//   fprop  Y[M,N]  = X[M,K] W[N,K]^T   A = X  (K-major), B = W (K-major)
//   dgrad  dX[M,K] = dY[M,N] W[N,K]    A = dY (K-major), B = W (MN-major)
//   wgrad  G[N,K] += dY^T X            A = dY (MN-major), B = X (MN-major), contraction M
// The wgrad contraction may be split across CTAs to fill the machine; the partial
// tiles meet in main_grad through the TMA fp32 reduce-add, the same in-place
// accumulation that the fused wgrad performs across microbatches.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>

#include "device.h"
#include "nv_block.cuh"
#include "sm100_ptx.cuh"
#include "tensor_map.h"

namespace gtp {
gtp_status launch_zero_bytes(void *data, int64_t nbytes, cudaStream_t stream, int sm_count);
}

__device__ unsigned int g_gtp_wait_timeouts;

namespace {

using namespace gtp::ptx;

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

enum { kStoreBf16 = 0, kReduceAddF32 = 1 };

struct Problem {
  int32_t m_dim, n_dim, k_dim;  // D rows, D columns, contraction length
  int32_t tiles_m, tiles_n, k_blocks, splits, num_units, group_m;
};

__device__ __forceinline__ void decode_unit(const Problem &p, int u, int &tm, int &tn, int &kb0, int &kb1) {
  const int split = u % p.splits;
  const int t = u / p.splits;
  const int per_group = p.group_m * p.tiles_n;
  const int g = t / per_group;
  const int first_m = g * p.group_m;
  const int gm = min(p.group_m, p.tiles_m - first_m);
  const int r = t - g * per_group;
  tm = first_m + r % gm;
  tn = r / gm;
  kb0 = int((int64_t(split) * p.k_blocks) / p.splits);
  kb1 = int((int64_t(split + 1) * p.k_blocks) / p.splits);
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

template <bool A_MN, bool B_MN, int EPI>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmD, const Problem p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + STAGES * A_STAGE;
  uint8_t *sEpi = smem + SMEM_OPERANDS;
  uint64_t *full = reinterpret_cast<uint64_t *>(sEpi + SMEM_EPI);
  uint64_t *empty = full + STAGES;
  uint64_t *tfull = empty + STAGES;
  uint64_t *tempty = tfull + 2;
  uint64_t *drain = tempty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], EPI_WARPS);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmD);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  unsigned int *err = &g_gtp_wait_timeouts;
  allow_dependents();  // set-up done: the next kernel may start launching into freed SMs
  wait_prior_grid();   // every global access below sees the previous kernel's results

  if (warp == 0) {
    if (lane == 0) {  // ---------------------------------------------------- TMA producer
      int stage = 0;
      uint32_t phase = 0;
      int armed[STAGES];
      for (int s = 0; s < STAGES; ++s) armed[s] = -1;
      for (int u = blockIdx.x; u < p.num_units; u += gridDim.x) {
        int tm, tn, kb0, kb1;
        decode_unit(p, u, tm, tn, kb0, kb1);
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, err, 0x1u)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
          armed[stage] = int(phase);
          uint8_t *a = sA + stage * A_STAGE;
          uint8_t *b = sB + stage * B_STAGE;
          const int k0 = kb * BK;
          if (A_MN) {
            tma_load_2d(&tmA, &full[stage], a, tm * BM, k0);
            tma_load_2d(&tmA, &full[stage], a + MN_CHUNK, tm * BM + 64, k0);
          } else {
            tma_load_2d(&tmA, &full[stage], a, k0, tm * BM);
          }
          if (B_MN) {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j) tma_load_2d(&tmB, &full[stage], b + j * MN_CHUNK, tn * BN + 64 * j, k0);
          } else {
            tma_load_2d(&tmB, &full[stage], b, k0, tn * BN);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      for (int s = 0; s < STAGES; ++s)  // every armed copy has landed before the CTA exits
        if (armed[s] >= 0) drain_wait(&full[s], uint32_t(armed[s]));
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---------------------------------------------------- MMA issuer
      const uint32_t idesc = idesc_bf16_f32(BM, BN, A_MN, B_MN);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
        int tm, tn, kb0, kb1;
        decode_unit(p, u, tm, tn, kb0, kb1);
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, err, 0x2u)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + uint32_t(acc * BN);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, err, 0x4u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * A_STAGE);
          const uint32_t b0 = smem_u32(sB + stage * B_STAGE);
#pragma unroll
          for (int k = 0; k < BK / UK; ++k) {
            const uint64_t ad = A_MN ? sdesc_sw128(a0 + k * (UK * 128), MN_CHUNK, 1024)
                                     : sdesc_sw128(a0 + k * (UK * 2), 16, 1024);
            const uint64_t bd = B_MN ? sdesc_sw128(b0 + k * (UK * 128), MN_CHUNK, 1024)
                                     : sdesc_sw128(b0 + k * (UK * 2), 16, 1024);
            mma_f16(d, ad, bd, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
          }
          mma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      mma_commit(drain);  // every issued MMA has finished before tensor memory is freed
      drain_wait(drain, 0);
    }
  } else {  // -------------------------------------------------------------- epilogue
    const int ew = warp - 2;
    const int quarter = warp & 3;  // tensor-memory lanes 32*quarter .. +31 belong to this warp
    uint8_t *mybuf = sEpi + ew * 2 * EPI_BUF;
    int acc = 0, bufsel = 0;
    uint32_t acc_phase = 0;
    constexpr int CW = (EPI == kStoreBf16) ? 64 : 32;  // columns per 128-byte staged row
    for (int u = blockIdx.x; u < p.num_units; u += gridDim.x) {
      int tm, tn, kb0, kb1;
      decode_unit(p, u, tm, tn, kb0, kb1);
      if (!mbar_wait(&tfull[acc], acc_phase, abort_flag, err, 0x8u)) break;
      tc_fence_after();
      const int row = tm * BM + 32 * quarter;
      const uint32_t tbase = tmem_base + (uint32_t(32 * quarter) << 16) + uint32_t(acc * BN);
#pragma unroll 1
      for (int c = 0; c < BN / CW; ++c) {
        uint32_t r0[32], r1[32];
        tmem_ld_32x32b_x32(tbase + uint32_t(c * CW), r0);
        if (EPI == kStoreBf16) tmem_ld_32x32b_x32(tbase + uint32_t(c * CW + 32), r1);
        tmem_ld_wait();
        uint8_t *buf = mybuf + bufsel * EPI_BUF;
        if (lane == 0) bulk_wait_group_read<1>();  // the store that last used `buf` has read it
        __syncwarp();
        stage_rows<EPI>(buf, lane, r0, r1);
        fence_proxy_async_smem();
        __syncwarp();
        const int col = tn * BN + c * CW;
        if (lane == 0) {
          if (row < p.m_dim && col < p.n_dim) {
            if (EPI == kStoreBf16)
              tma_store_2d(&tmD, buf, col, row);
            else
              tma_reduce_add_2d(&tmD, buf, col, row);
          }
          bulk_commit_group();
        }
        bufsel ^= 1;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // the staging buffers must outlive the stores' reads of them; the global writes
    // themselves complete with the grid, which is what a stream or a dependent grid waits for
    if (lane == 0) bulk_wait_group_read<0>();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// --------------------------------------------------------------------------- CTA-pair GEMM
//
// The same product on a pair of CTAs (a cluster of two SMs) sharing one tcgen05.mma of
// M = 256, N = 256 (cta_group::2).  Each CTA stages 128 rows of A and 128 rows of B per
// k-block (32 KB), half of what a 128x256 single-CTA tile needs per MMA, and holds its
// 128 x 256 rows of D in its own tensor memory.  Shared-memory traffic per SM drops from
// 12 KB to 8 KB per 128 tensor cycles, which the single-CTA tile is bound by.
//   Both CTAs' TMA copies complete on the even CTA's full[] barrier (cta_group::2 loads),
//   which the even CTA arms for the bytes of both halves; its warp 1 issues the MMAs and
//   multicasts the commits to both CTAs' empty[] / tfull[].  The epilogue warps of both
//   CTAs release an accumulator on the even CTA's tempty[].  At exit the even CTA drains
//   every stage it armed (the odd CTA's copies included) before the closing cluster
//   barrier, so neither CTA leaves with a copy in flight.
//   Work distribution (DYN): the grid holds one cluster per work unit.  A running pair
//   starts with its own unit; the even CTA's producer thread then asks the hardware to
//   cancel a cluster that has not started yet (cluster launch control) and the pair takes
//   over that cluster's unit.  Each 16-byte response lands in both CTAs' shared memory
//   (an 8-slot ring); every role of both CTAs reads the responses in order and releases a
//   slot on the even CTA's clc_empty[].  Pairs that run faster take more units, which a
//   static round-robin assignment cannot do.  Without DYN the pairs take units
//   cluster, cluster + nclusters, ... of a grid of at most one wave.
namespace pair {
constexpr int BMP = 256;       // rows of a pair tile
constexpr int BMC = 128;       // rows per CTA
constexpr int BNC = 128;       // B rows staged per CTA (the pair tile has BN = 256 columns)
constexpr int STAGES = 6;
constexpr int A_STAGE = BMC * BK * 2;  // 16 KB
constexpr int B_STAGE = BNC * BK * 2;  // 16 KB
constexpr int STAGE_BYTES = A_STAGE + B_STAGE;
constexpr int SMEM_OPS = STAGES * STAGE_BYTES;
constexpr int SCHED = 8;               // cancel responses in flight
constexpr uint32_t SCHED_CONSUMERS = 12;  // per CTA: producer, warp-1 lane 0, 4 epilogue warps
constexpr int CTRL = 512;
constexpr int SMEM_TOTAL = SMEM_OPS + SMEM_EPI + CTRL + 1024;
static_assert(SMEM_TOTAL <= 232448, "shared memory per block");
static_assert(16 * SCHED + (2 * STAGES + 5 + 2 * SCHED) * 8 + 8 <= CTRL, "control block");
}  // namespace pair

// The next work unit of a role of a CTA pair, or -1 when none is left.  Dynamic: waits for
// the response in the role's current ring slot, decodes it and releases the slot.
template <bool DYN>
__device__ __forceinline__ int advance_unit(int unit, int &slot, uint32_t &phase, int nclusters, const Problem &p,
                                            const uint8_t *resp, uint64_t *clc_full, uint64_t *clc_empty,
                                            volatile int *abort_flag, unsigned int *err) {
  if (!DYN) {
    unit += nclusters;
    return unit < p.num_units ? unit : -1;
  }
  if (!mbar_wait(&clc_full[slot], phase, abort_flag, err, 0x20u)) return -1;
  uint32_t x = 0;
  const bool ok = clc_decode(resp + 16 * slot, x);
  mbar_arrive_cluster(mapa_shared(&clc_empty[slot], 0));
  if (++slot == pair::SCHED) {
    slot = 0;
    phase ^= 1u;
  }
  if (!ok) return -1;
  const int u = int(x >> 1);  // clusters are pairs of consecutive CTAs: cluster = first CTA / 2
  return u < p.num_units ? u : -1;
}

// Dynamic scheduling: prepares the ring slot that will carry the next response.  Both CTAs'
// producers arm their own clc_full[slot] for 16 bytes; the even CTA's producer, once every
// role of both CTAs has released the slot, issues the cancel request.
__device__ __forceinline__ bool clc_request(bool leader, int slot, uint32_t phase, uint8_t *resp, uint64_t *clc_full,
                                            uint64_t *clc_empty, volatile int *abort_flag, unsigned int *err) {
  if (leader && !mbar_wait(&clc_empty[slot], phase ^ 1u, abort_flag, err, 0x40u)) return false;
  mbar_arrive_expect_tx(&clc_full[slot], 16);
  if (leader) clc_try_cancel_multicast(resp + 16 * slot, &clc_full[slot]);
  return true;
}

template <bool A_MN, bool B_MN, int EPI, bool DYN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    gemm_bf16_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmD, const Problem p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + pair::STAGES * pair::A_STAGE;
  uint8_t *sEpi = smem + pair::SMEM_OPS;
  uint8_t *resp = sEpi + SMEM_EPI;  // 16-byte cancel responses, SCHED slots
  uint64_t *full = reinterpret_cast<uint64_t *>(resp + 16 * pair::SCHED);
  uint64_t *empty = full + pair::STAGES;
  uint64_t *tfull = empty + pair::STAGES;
  uint64_t *tempty = tfull + 2;
  uint64_t *drain = tempty + 2;
  uint64_t *clc_full = drain + 1;
  uint64_t *clc_empty = clc_full + pair::SCHED;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(clc_empty + pair::SCHED);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cluster = int(blockIdx.x >> 1), nclusters = int(gridDim.x >> 1);
  if (threadIdx.x == 0) {
    for (int s = 0; s < pair::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * EPI_WARPS);
    }
    mbar_init(drain, 1);
    for (int s = 0; s < pair::SCHED; ++s) {
      mbar_init(&clc_full[s], 1);
      mbar_init(&clc_empty[s], pair::SCHED_CONSUMERS);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmD);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any remote arrive or multicast
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  unsigned int *err = &g_gtp_wait_timeouts;
  allow_dependents();  // set-up done: the next kernel may start launching into freed SMs
  wait_prior_grid();   // every global access below sees the previous kernel's results
  const int first = cluster < p.num_units ? cluster : -1;

  if (warp == 0) {
    if (lane == 0) {  // ------------------------------------------ TMA producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0;
      int armed[pair::STAGES];
      for (int s = 0; s < pair::STAGES; ++s) armed[s] = -1;
      int slot = 0;
      uint32_t sphase = 0;
      int unit = first;
      if (DYN && unit >= 0 && !clc_request(rank == 0, slot, sphase, resp, clc_full, clc_empty, abort_flag, err))
        unit = -1;
      while (unit >= 0) {
        int tm, tn, kb0, kb1;
        decode_unit(p, unit, tm, tn, kb0, kb1);
        const int m0 = tm * pair::BMP + pair::BMC * int(rank);
        const int n0 = tn * BN + pair::BNC * int(rank);
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, err, 0x1u)) {
            ok = false;
            break;
          }
          if (rank == 0) {  // the even CTA's barrier counts both CTAs' bytes
            mbar_arrive_expect_tx(&full[stage], 2 * pair::STAGE_BYTES);
            armed[stage] = int(phase);
          }
          const uint32_t bar = mapa_shared(&full[stage], 0);
          uint8_t *a = sA + stage * pair::A_STAGE;
          uint8_t *b = sB + stage * pair::B_STAGE;
          const int k0 = kb * BK;
          if (A_MN) {
            tma_load_2d_pair(&tmA, bar, a, m0, k0);
            tma_load_2d_pair(&tmA, bar, a + MN_CHUNK, m0 + 64, k0);
          } else {
            tma_load_2d_pair(&tmA, bar, a, k0, m0);
          }
          if (B_MN) {
            tma_load_2d_pair(&tmB, bar, b, n0, k0);
            tma_load_2d_pair(&tmB, bar, b + MN_CHUNK, n0 + 64, k0);
          } else {
            tma_load_2d_pair(&tmB, bar, b, k0, n0);
          }
          if (++stage == pair::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        unit = advance_unit<DYN>(unit, slot, sphase, nclusters, p, resp, clc_full, clc_empty, abort_flag, err);
        if (DYN && unit >= 0 && !clc_request(rank == 0, slot, sphase, resp, clc_full, clc_empty, abort_flag, err))
          break;
      }
      for (int s = 0; s < pair::STAGES; ++s)
        if (armed[s] >= 0) drain_wait(&full[s], uint32_t(armed[s]));
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ----------- MMA issuer (even CTA); the odd CTA only follows the units
      const uint32_t idesc = idesc_bf16_f32(pair::BMP, BN, A_MN, B_MN);
      int stage = 0, acc = 0, slot = 0;
      uint32_t phase = 0, acc_phase = 0, sphase = 0;
      int unit = first;
      while (unit >= 0) {
        if (rank == 0) {
          int tm, tn, kb0, kb1;
          decode_unit(p, unit, tm, tn, kb0, kb1);
          if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, err, 0x2u)) break;
          tc_fence_after();
          const uint32_t d = tmem_base + uint32_t(acc * BN);
          bool ok = true;
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait(&full[stage], phase, abort_flag, err, 0x4u)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(sA + stage * pair::A_STAGE);
            const uint32_t b0 = smem_u32(sB + stage * pair::B_STAGE);
#pragma unroll
            for (int k = 0; k < BK / UK; ++k) {
              const uint64_t ad = A_MN ? sdesc_sw128(a0 + k * (UK * 128), MN_CHUNK, 1024)
                                       : sdesc_sw128(a0 + k * (UK * 2), 16, 1024);
              const uint64_t bd = B_MN ? sdesc_sw128(b0 + k * (UK * 128), MN_CHUNK, 1024)
                                       : sdesc_sw128(b0 + k * (UK * 2), 16, 1024);
              mma_f16_pair(d, ad, bd, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
            }
            mma_commit_pair(&empty[stage], 0x3);
            if (++stage == pair::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit_pair(&tfull[acc], 0x3);
          if (++acc == 2) {
            acc = 0;
            acc_phase ^= 1u;
          }
        }
        unit = advance_unit<DYN>(unit, slot, sphase, nclusters, p, resp, clc_full, clc_empty, abort_flag, err);
      }
      if (rank == 0) mma_commit_pair(drain, 0x3);  // both CTAs learn when every MMA has finished
      drain_wait(drain, 0);
    }
  } else {  // -------------------------------------------------------- epilogue (both CTAs)
    const int ew = warp - 2;
    const int quarter = warp & 3;
    uint8_t *mybuf = sEpi + ew * 2 * EPI_BUF;
    int acc = 0, bufsel = 0, slot = 0;
    uint32_t acc_phase = 0, sphase = 0;
    constexpr int CW = (EPI == kStoreBf16) ? 64 : 32;
    int unit = first;
    while (unit >= 0) {
      int tm, tn, kb0, kb1;
      decode_unit(p, unit, tm, tn, kb0, kb1);
      const bool ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, err, 0x8u);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;  // the warp leaves together
      tc_fence_after();
      const int row = tm * pair::BMP + pair::BMC * int(rank) + 32 * quarter;
      const uint32_t tbase = tmem_base + (uint32_t(32 * quarter) << 16) + uint32_t(acc * BN);
#pragma unroll 1
      for (int c = 0; c < BN / CW; ++c) {
        uint32_t r0[32], r1[32];
        tmem_ld_32x32b_x32(tbase + uint32_t(c * CW), r0);
        if (EPI == kStoreBf16) tmem_ld_32x32b_x32(tbase + uint32_t(c * CW + 32), r1);
        tmem_ld_wait();
        uint8_t *buf = mybuf + bufsel * EPI_BUF;
        if (lane == 0) bulk_wait_group_read<1>();
        __syncwarp();
        stage_rows<EPI>(buf, lane, r0, r1);
        fence_proxy_async_smem();
        __syncwarp();
        const int col = tn * BN + c * CW;
        if (lane == 0) {
          if (row < p.m_dim && col < p.n_dim) {
            if (EPI == kStoreBf16)
              tma_store_2d(&tmD, buf, col, row);
            else
              tma_reduce_add_2d(&tmD, buf, col, row);
          }
          bulk_commit_group();
        }
        bufsel ^= 1;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(&tempty[acc], 0));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
      int next = -1;
      if (lane == 0)
        next = advance_unit<DYN>(unit, slot, sphase, nclusters, p, resp, clc_full, clc_empty, abort_flag, err);
      unit = __shfl_sync(0xFFFFFFFFu, next, 0);
    }
    // the staging buffers must outlive the stores' reads of them; the global writes
    // themselves complete with the grid, which is what a stream or a dependent grid waits for
    if (lane == 0) bulk_wait_group_read<0>();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the other may still reach its shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------ block-scaled (MXFP8, NVFP4)
//
// Y[M,N] (bf16) = dq(Xq, Xs) dq(Wq, Ws)^T on the block-scaled tensor-core path, operands
// K-major with 128-byte rows per stage, scales read from tensor memory:
//   MXFP8  kind::mxf8f6f4.block_scale.scale_vec::1X: E4M3 elements, one E8M0 scale per
//          32; a stage holds 128 K (one 32-bit scale word per row: 4 blocks, and the MMA
//          of K block k reads byte k of it through the sf_id field);
//   NVFP4  kind::mxf4nvf4.block_scale.scale_vec::4X: packed E2M1 elements, one E4M3
//          scale per 16; a stage holds 256 K (four scale words per row, one per MMA of
//          K 64), and the epilogue multiplies by 1 / (S_A S_B), the per-tensor scales.
// The scales arrive in the natural [rows, K/block] byte layout; the producer warp
// gathers, per stage, each row's scale words and writes them where
// tcgen05.cp.32x128b.warpx4 expects them: for every 128 rows and word w, the word of row
// 32*c + l at word index 4*l + c, so that tensor-memory lane r finds its row's word in
// column r / 32 of the word's 4-column group (8 columns for the 256 B rows).
//   tensor memory: columns [0, 256) fp32 accumulator, then the A scale groups (4 columns
//   per word and stage), then the B scale groups (8 columns per word and stage).
enum { kMxfp8 = 0, kNvfp4 = 1 };

// The block-scaled kernel keeps one accumulator (the scale columns take the rest of tensor
// memory), so its epilogue runs 8 warps, two per 32-lane quarter, each holding half of its
// rows' 256 columns in registers: the accumulator is released as soon as it has been read,
// and the conversion and stores of one tile overlap the main loop of the next.
constexpr int kBsEpiWarps = 8;
constexpr int kBsThreads = 64 + 32 * kBsEpiWarps;

constexpr int kBsEpiBuf = 32 * 64;  // per epilogue warp: 32 rows x 64 bytes (64-byte swizzle)

// S: operand stages.  The ring is what keeps loads in flight, so the staging buffers stay
// small to leave room for it; but shared memory also sets the L1 size left over, and a
// long contraction re-reads each row's scale words from L1 stage after stage.  MXFP8 runs
// 4 stages on short contractions and 3 on long ones (the host picks); NVFP4, whose scale
// words take 6 KB per stage, always runs 3.
template <int FMT, int S = 3>
struct BlockScaled {
  static constexpr int STAGES = S;
  static constexpr int WORDS = FMT == kMxfp8 ? 1 : 4;       // scale words per row per stage
  static constexpr int K_STAGE = FMT == kMxfp8 ? 128 : 256;  // K elements per stage
  static constexpr int BK = 128;                             // code bytes per row per stage
  static constexpr int UKB = 32;                             // code bytes per instruction
  static constexpr int SF_BLOCK = FMT == kMxfp8 ? 32 : 16;   // K elements per scale
  static constexpr int A_STAGE = BM * BK;                    // 16 KB
  static constexpr int B_STAGE = BN * BK;                    // 32 KB
  static constexpr int SFA_STAGE = BM * 4 * WORDS;
  static constexpr int SFB_STAGE = BN * 4 * WORDS;
  static constexpr int STAGE_TX = A_STAGE + B_STAGE;
  static constexpr int SMEM_OPS = STAGES * (A_STAGE + B_STAGE);
  // padded to 1 KB: the epilogue staging buffers that follow must start on the 1024-byte
  // period of the 128-byte swizzle the output tensor map uses
  static constexpr int SMEM_SF = (STAGES * (SFA_STAGE + SFB_STAGE) + 1023) / 1024 * 1024;
  static_assert((STAGES * (A_STAGE + B_STAGE) + SMEM_SF) % 1024 == 0, "staging buffers 1024-byte aligned");
  static constexpr int SMEM_EPI = kBsEpiWarps * kBsEpiBuf;  // one staging buffer per epilogue warp
  static constexpr int SMEM_TOTAL = SMEM_OPS + SMEM_SF + SMEM_EPI + SMEM_CTRL + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t SFA_COL = BN;
  static constexpr uint32_t SFB_COL = BN + 4 * WORDS * STAGES;
  static constexpr int PREFETCH = FMT == kMxfp8 ? 4 : 2;  // stages of scale words in registers
  static_assert(SMEM_TOTAL <= 232448, "shared memory per block");
  static_assert(SFB_COL + 8 * WORDS * STAGES <= TMEM_COLS, "tensor memory columns");
};

// One stage of a lane's scale words: A rows 32c + lane (c < 4) and B rows 128j + 32c + lane
// (index 4j + c), WORDS words each.
template <int WORDS>
struct ScaleRegs {
  uint32_t a[4][WORDS];
  uint32_t b[8][WORDS];
};

// Walks one CTA's (unit, k-block) sequence of the static round-robin schedule.
struct StageIter {
  int u, tm, tn, kb, kb1;
  __device__ __forceinline__ void start(const Problem &p, int unit) {
    u = unit;
    if (u < p.num_units) decode_unit(p, u, tm, tn, kb, kb1);
  }
  __device__ __forceinline__ bool valid(const Problem &p) const { return u < p.num_units; }
  __device__ __forceinline__ void next(const Problem &p) {
    if (++kb == kb1) start(p, u + int(gridDim.x));
  }
};

template <int WORDS>
__device__ __forceinline__ void load_row_words(uint32_t (&w)[WORDS], const uint8_t *sf, int64_t row_bytes, int r,
                                               int rows, int kb) {
  const uint8_t *row = sf + int64_t(r) * row_bytes;
  if (WORDS == 4) {  // 16 bytes per row and stage: one vector load (16-byte aligned rows)
    const uint4 v = r < rows ? __ldg(reinterpret_cast<const uint4 *>(row) + kb) : make_uint4(0u, 0u, 0u, 0u);
    w[0] = v.x;
    w[1 % WORDS] = v.y;
    w[2 % WORDS] = v.z;
    w[3 % WORDS] = v.w;
  } else {
    w[0] = r < rows ? __ldg(reinterpret_cast<const uint32_t *>(row) + kb) : 0u;
  }
}

template <int WORDS>
__device__ __forceinline__ void load_scales(ScaleRegs<WORDS> &R, const uint8_t *sfa, const uint8_t *sfb,
                                            int64_t row_bytes, const Problem &p, int tm, int tn, int kb, int lane) {
#pragma unroll
  for (int c = 0; c < 4; ++c) load_row_words<WORDS>(R.a[c], sfa, row_bytes, tm * BM + 32 * c + lane, p.m_dim, kb);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    load_row_words<WORDS>(R.b[i], sfb, row_bytes, tn * BN + 128 * (i >> 2) + 32 * (i & 3) + lane, p.n_dim, kb);
}

// Word w of a stage, for each group of 128 rows, goes where tcgen05.cp.32x128b.warpx4
// expects it: the word of row 32c + l at word index 4l + c of the group's 128 words.
template <int WORDS>
__device__ __forceinline__ void store_scales(const ScaleRegs<WORDS> &R, uint32_t *fa, uint32_t *fb, int lane) {
#pragma unroll
  for (int w = 0; w < WORDS; ++w) {
    *reinterpret_cast<uint4 *>(fa + 128 * w + 4 * lane) = make_uint4(R.a[0][w], R.a[1][w], R.a[2][w], R.a[3][w]);
#pragma unroll
    for (int j = 0; j < 2; ++j)
      *reinterpret_cast<uint4 *>(fb + 128 * (2 * w + j) + 4 * lane) =
          make_uint4(R.b[4 * j][w], R.b[4 * j + 1][w], R.b[4 * j + 2][w], R.b[4 * j + 3][w]);
  }
}

// EPI: kStoreBf16 (fprop, dgrad) or kReduceAddF32 (wgrad into the fp32 main_grad view).
// a_amax, b_amax: the NVFP4 tensor amaxes (device scalars; unused for MXFP8).
template <int FMT, int EPI, int S>
__global__ void __launch_bounds__(kBsThreads, 1)
    gemm_blockscaled_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmD, const uint8_t *__restrict__ sfa_g,
                            const uint8_t *__restrict__ sfb_g, const float *__restrict__ a_amax,
                            const float *__restrict__ b_amax, const Problem p) {
  using F = BlockScaled<FMT, S>;
  constexpr int STAGES = F::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sA = smem;
  uint8_t *sB = sA + STAGES * F::A_STAGE;
  uint32_t *sSFA = reinterpret_cast<uint32_t *>(smem + F::SMEM_OPS);
  uint32_t *sSFB = sSFA + STAGES * (F::SFA_STAGE / 4);
  uint8_t *sEpi = smem + F::SMEM_OPS + F::SMEM_SF;
  uint64_t *full = reinterpret_cast<uint64_t *>(sEpi + F::SMEM_EPI);
  uint64_t *empty = full + STAGES;
  uint64_t *tfull = empty + STAGES;
  uint64_t *tempty = tfull + 1;
  uint64_t *drain = tempty + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, kBsEpiWarps);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmD);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, F::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  unsigned int *err = &g_gtp_wait_timeouts;
  allow_dependents();  // set-up done: the next kernel may start launching into freed SMs
  wait_prior_grid();   // every global access below sees the previous kernel's results
  const int64_t sf_row_bytes = p.k_dim / F::SF_BLOCK;

  if (warp == 0) {  // ------------------------------------------------------ producer warp
    int stage = 0;
    uint32_t phase = 0;
    int armed[STAGES];
    for (int s = 0; s < STAGES; ++s) armed[s] = -1;
    // The scale words of the next PREFETCH stages sit in registers (a ring indexed by the
    // unrolled d), so a stage's global-load latency overlaps the stages before it.
    constexpr int D = F::PREFETCH;
    ScaleRegs<F::WORDS> ring[D];
    StageIter ld, st;
    ld.start(p, blockIdx.x);
    st = ld;
#pragma unroll
    for (int d = 0; d < D; ++d)
      if (ld.valid(p)) {
        load_scales(ring[d], sfa_g, sfb_g, sf_row_bytes, p, ld.tm, ld.tn, ld.kb, lane);
        ld.next(p);
      }
    bool ok = true;
    while (ok && st.valid(p)) {
#pragma unroll
      for (int d = 0; d < D; ++d) {
        if (!st.valid(p)) break;
        int got = 1;
        if (lane == 0) got = mbar_wait(&empty[stage], phase ^ 1u, abort_flag, err, 0x1u) ? 1 : 0;
        got = __shfl_sync(0xFFFFFFFFu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        store_scales(ring[d], sSFA + stage * (F::SFA_STAGE / 4), sSFB + stage * (F::SFB_STAGE / 4), lane);
        fence_proxy_async_smem();  // the scale words are read by tcgen05.cp (async proxy)
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[stage], F::STAGE_TX);
          armed[stage] = int(phase);
          tma_load_2d(&tmA, &full[stage], sA + stage * F::A_STAGE, st.kb * F::BK, st.tm * BM);
          tma_load_2d(&tmB, &full[stage], sB + stage * F::B_STAGE, st.kb * F::BK, st.tn * BN);
        }
        if (ld.valid(p)) {
          load_scales(ring[d], sfa_g, sfb_g, sf_row_bytes, p, ld.tm, ld.tn, ld.kb, lane);
          ld.next(p);
        }
        st.next(p);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (lane == 0)
      for (int s = 0; s < STAGES; ++s)
        if (armed[s] >= 0) drain_wait(&full[s], uint32_t(armed[s]));
  } else if (warp == 1) {
    if (lane == 0) {  // ---------------------------------------------------- MMA issuer
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
        int tm, tn, kb0, kb1;
        decode_unit(p, u, tm, tn, kb0, kb1);
        if (!mbar_wait(tempty, acc_phase ^ 1u, abort_flag, err, 0x2u)) break;
        tc_fence_after();
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, err, 0x4u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfa_t = tmem_base + F::SFA_COL + 4 * F::WORDS * stage;
          const uint32_t sfb_t = tmem_base + F::SFB_COL + 8 * F::WORDS * stage;
          const uint32_t *fa = sSFA + stage * (F::SFA_STAGE / 4);
          const uint32_t *fb = sSFB + stage * (F::SFB_STAGE / 4);
#pragma unroll
          for (int w = 0; w < F::WORDS; ++w) {
            tmem_cp_32x128b_warpx4(sfa_t + 4 * w, sdesc_noswizzle_rows16(smem_u32(fa + 128 * w)));
            tmem_cp_32x128b_warpx4(sfb_t + 8 * w, sdesc_noswizzle_rows16(smem_u32(fb + 128 * (2 * w))));
            tmem_cp_32x128b_warpx4(sfb_t + 8 * w + 4, sdesc_noswizzle_rows16(smem_u32(fb + 128 * (2 * w + 1))));
          }
          const uint32_t a0 = smem_u32(sA + stage * F::A_STAGE);
          const uint32_t b0 = smem_u32(sB + stage * F::B_STAGE);
#pragma unroll
          for (int k = 0; k < F::BK / F::UKB; ++k) {
            const uint64_t ad = sdesc_sw128(a0 + k * F::UKB, 16, 1024);
            const uint64_t bd = sdesc_sw128(b0 + k * F::UKB, 16, 1024);
            const uint32_t acc = (kb > kb0 || k > 0) ? 1u : 0u;
            if (FMT == kMxfp8)  // byte k of the stage's scale word
              mma_mxf8_block_scale(tmem_base, ad, bd, idesc_mxf8_e4m3(BM, BN, uint32_t(k)), sfa_t, sfb_t, acc);
            else  // scale word k: the four 16-blocks of this instruction's 64 K
              mma_nvf4_block_scale(tmem_base, ad, bd, idesc_nvf4_e2m1(BM, BN), sfa_t + 4 * k, sfb_t + 8 * k, acc);
          }
          mma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(tfull);
        acc_phase ^= 1u;
      }
      mma_commit(drain);
      drain_wait(drain, 0);
    }
  } else {  // -------------------------------------------------------------- epilogue
    // warp w reads tensor-memory lanes 32 (w % 4) .. +31 (the quarter a warp may access)
    // and columns 128 h .. +127 of them, h = (w - 2) / 4
    const int ew = warp - 2;
    const int quarter = warp & 3;
    const int half = ew >> 2;
    uint8_t *buf = sEpi + ew * kBsEpiBuf;
    uint32_t acc_phase = 0;
    // NVFP4: the MMA applied the block scales; the per-tensor ones leave as 1 / (S_A S_B)
    float alpha = 1.f;
    if (FMT == kNvfp4)
      alpha = float(1.0 / (double(gtp::nv::tensor_scale(__ldg(a_amax))) * double(gtp::nv::tensor_scale(__ldg(b_amax)))));
    for (int u = blockIdx.x; u < p.num_units; u += gridDim.x) {
      int tm, tn, kb0, kb1;
      decode_unit(p, u, tm, tn, kb0, kb1);
      if (!mbar_wait(tfull, acc_phase, abort_flag, err, 0x8u)) break;
      tc_fence_after();
      const int row = tm * BM + 32 * quarter;
      const uint32_t tbase = tmem_base + (uint32_t(32 * quarter) << 16) + uint32_t(half * (BN / 2));
      uint32_t r[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(tbase + uint32_t(32 * c), r[c]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty);  // the next tile's MMAs may overwrite the accumulator
      if (FMT == kNvfp4) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) r[c][i] = __float_as_uint(__uint_as_float(r[c][i]) * alpha);
      }
      constexpr int CW = (EPI == kStoreBf16) ? 32 : 16;  // columns per 64-byte staged row
#pragma unroll
      for (int q = 0; q < (BN / 2) / CW; ++q) {
        if (lane == 0) bulk_wait_group_read<0>();  // the previous store has read `buf`
        __syncwarp();
        if (EPI == kStoreBf16)
          stage_rows64<EPI>(buf, lane, r[q], 0);
        else
          stage_rows64<EPI>(buf, lane, r[q >> 1], 16 * (q & 1));
        fence_proxy_async_smem();
        __syncwarp();
        const int col = tn * BN + half * (BN / 2) + q * CW;
        if (lane == 0) {
          if (row < p.m_dim && col < p.n_dim) {
            if (EPI == kStoreBf16)
              tma_store_2d(&tmD, buf, col, row);
            else
              tma_reduce_add_2d(&tmD, buf, col, row);
          }
          bulk_commit_group();
        }
      }
      acc_phase ^= 1u;
    }
    // the staging buffers must outlive the stores' reads of them; the global writes
    // themselves complete with the grid, which is what a stream or a dependent grid waits for
    if (lane == 0) bulk_wait_group_read<0>();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, F::TMEM_COLS);
  }
}

// --------------------------------------------------------------------------- host side

int choose_splits(int tiles, int k_blocks, int sms) {
  int best = 1;
  double best_score = -1.0;
  for (int s = 1; s <= 8 && s <= k_blocks; ++s) {
    if (s > 1 && k_blocks / s < 4) break;
    const int64_t units = int64_t(tiles) * s;
    const int64_t waves = (units + sms - 1) / sms;
    const double score = double(units) / double(waves * sms) - 0.03 * (s - 1);
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

// Which kernel serves a problem: the CTA pair unless the output has at most 128 rows
// (half of every pair tile would be empty).  The environment variable
// GTP_GEMM_VARIANT=single|pair overrides the choice (read at each call; the tests use it
// to cover both kernels).
bool use_pair(int m_dim) {
  if (const char *v = std::getenv("GTP_GEMM_VARIANT")) {
    if (!std::strcmp(v, "single")) return false;
    if (!std::strcmp(v, "pair")) return true;
  }
  return m_dim > BM;
}

template <typename K>
gtp_status configure(K kernel, int smem, std::atomic<uint64_t> &configured, int device) {
  const uint64_t bit = uint64_t(1) << (device & 63);
  if (configured.load() & bit) return GTP_OK;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return gtp::fail(GTP_E_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  configured.fetch_or(bit);
  return GTP_OK;
}

// Co-resident CTA pairs of the pair kernel on the current device (cached per device).
template <typename K>
int max_pairs(K kernel, const gtp::DeviceInfo &dev) {
  static std::atomic<int> cached[64];
  int v = cached[dev.device & 63].load();
  if (v > 0) return v;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(dev.sm_count & ~1));
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = pair::SMEM_TOTAL;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = dev.sm_count / 2;
  }
  cached[dev.device & 63].store(n);
  return n;
}

// A (rows x k) and B (cols x k) operands, K-major (contraction contiguous) or MN-major
// (rows / cols contiguous, one row of memory per contraction index); D (m_dim x n_dim)
// row-major bf16 (store) or fp32 (reduce-add).
struct Operands {
  const void *a, *b;
  void *d;
  int m_dim, n_dim, k_dim;
};

template <bool A_MN, bool B_MN, int EPI>
gtp_status run_gemm(const Operands &o, bool allow_split, const gtp::DeviceInfo &dev, cudaStream_t stream) {
  const bool pr = use_pair(o.m_dim);
  const int bm = pr ? pair::BMP : BM;
  const uint32_t b_rows = pr ? pair::BNC : BN;  // B rows staged per CTA
  CUtensorMap ta, tb, td;
  gtp_status s;
  if (A_MN)
    s = gtp::encode_tmap_2d(&ta, kBF16, o.a, o.m_dim, o.k_dim, uint64_t(o.m_dim) * 2, 64, BK, kSW128);
  else
    s = gtp::encode_tmap_2d(&ta, kBF16, o.a, o.k_dim, o.m_dim, uint64_t(o.k_dim) * 2, 64, BM, kSW128);
  if (s) return s;
  if (B_MN)
    s = gtp::encode_tmap_2d(&tb, kBF16, o.b, o.n_dim, o.k_dim, uint64_t(o.n_dim) * 2, 64, BK, kSW128);
  else
    s = gtp::encode_tmap_2d(&tb, kBF16, o.b, o.k_dim, o.n_dim, uint64_t(o.k_dim) * 2, 64, b_rows, kSW128);
  if (s) return s;
  if (EPI == kStoreBf16)
    s = gtp::encode_tmap_2d(&td, kBF16, o.d, o.n_dim, o.m_dim, uint64_t(o.n_dim) * 2, 64, 32, kSW128);
  else
    s = gtp::encode_tmap_2d(&td, kF32, o.d, o.n_dim, o.m_dim, uint64_t(o.n_dim) * 4, 32, 32, kSW128);
  if (s) return s;
  Problem p;
  p.m_dim = o.m_dim;
  p.n_dim = o.n_dim;
  p.k_dim = o.k_dim;
  p.tiles_m = (o.m_dim + bm - 1) / bm;
  p.tiles_n = (o.n_dim + BN - 1) / BN;
  p.k_blocks = (o.k_dim + BK - 1) / BK;
  p.group_m = pr ? 8 : 16;
  const int tiles = p.tiles_m * p.tiles_n;
  if (pr) {
    // Round-robin one-wave grid by default; GTP_GEMM_SCHED=dynamic selects the
    // cluster-launch-control schedule (measured 2% slower over the layer step on GB300,
    // where the pairs' speeds turned out too even for it to pay off).
    const char *sched = std::getenv("GTP_GEMM_SCHED");
    const bool dyn = sched && !std::strcmp(sched, "dynamic");
    static std::atomic<uint64_t> configured_s{0}, configured_d{0};
    auto ks = gemm_bf16_pair_kernel<A_MN, B_MN, EPI, false>;
    auto kd = gemm_bf16_pair_kernel<A_MN, B_MN, EPI, true>;
    auto kernel = dyn ? kd : ks;
    if (gtp_status e = configure(kernel, pair::SMEM_TOTAL, dyn ? configured_d : configured_s, dev.device)) return e;
    const int pairs = max_pairs(ks, dev);
    p.splits = allow_split ? choose_splits(tiles, p.k_blocks, pairs) : 1;
    p.num_units = tiles * p.splits;
    const int grid = 2 * (dyn ? p.num_units : std::min(p.num_units, pairs));
    return gtp::launch_overlapped(kernel, grid, kGemmThreads, pair::SMEM_TOTAL, stream, "gemm_bf16_pair_kernel", ta,
                                  tb, td, p);
  }
  static std::atomic<uint64_t> configured{0};
  auto kernel = gemm_bf16_kernel<A_MN, B_MN, EPI>;
  if (gtp_status e = configure(kernel, SMEM_TOTAL, configured, dev.device)) return e;
  p.splits = allow_split ? choose_splits(tiles, p.k_blocks, dev.sm_count) : 1;
  p.num_units = tiles * p.splits;
  const int grid = std::min(p.num_units, dev.sm_count);
  return gtp::launch_overlapped(kernel, grid, kGemmThreads, SMEM_TOTAL, stream, "gemm_bf16_kernel", ta, tb, td, p);
}

constexpr int64_t kMaxDim = int64_t(1) << 30;

gtp_status check_dims(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 0) return gtp::fail(GTP_E_ARG, "negative dimension");
  if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return gtp::fail(GTP_E_SHAPE, "dimension above 2^30");
  if (N % 8 || K % 8) return gtp::fail(GTP_E_ALIGN, "N and K must be multiples of 8 (16-byte rows)");
  return GTP_OK;
}

}  // namespace

namespace gtp {
void clear_error();
}

extern "C" gtp_status gtp_linear_fprop(const void *X, const void *W, void *Y, int64_t M, int64_t N, int64_t K,
                                       gtp_dtype dt, gtp_stream stream) {
  gtp::clear_error();
  if (dt != GTP_BF16) return gtp::fail(GTP_E_DTYPE, "only GTP_BF16 is supported");
  if (gtp_status s = check_dims(M, N, K)) return s;
  if (M == 0 || N == 0) return GTP_OK;
  if (!Y || (K > 0 && (!X || !W))) return gtp::fail(GTP_E_ARG, "null pointer");
  if (!gtp::aligned16(Y) || (K > 0 && (!gtp::aligned16(X) || !gtp::aligned16(W))))
    return gtp::fail(GTP_E_ALIGN, "pointers must be 16-byte aligned");
  gtp::DeviceInfo dev;
  if (gtp_status s = gtp::require_sm103(&dev)) return s;
  cudaStream_t st = gtp::as_stream(stream);
  if (K == 0) return gtp::launch_zero_bytes(Y, M * N * 2, st, dev.sm_count);
  // D = Y [M, N]; A = X (K-major), B = W [N, K] (K-major)
  return run_gemm<false, false, kStoreBf16>({X, W, Y, int(M), int(N), int(K)}, false, dev, st);
}

extern "C" gtp_status gtp_linear_dgrad(const void *dY, const void *W, void *dX, int64_t M, int64_t N, int64_t K,
                                       gtp_dtype dt, gtp_stream stream) {
  gtp::clear_error();
  if (dt != GTP_BF16) return gtp::fail(GTP_E_DTYPE, "only GTP_BF16 is supported");
  if (gtp_status s = check_dims(M, N, K)) return s;
  if (M == 0 || K == 0) return GTP_OK;
  if (!dX || (N > 0 && (!dY || !W))) return gtp::fail(GTP_E_ARG, "null pointer");
  if (!gtp::aligned16(dX) || (N > 0 && (!gtp::aligned16(dY) || !gtp::aligned16(W))))
    return gtp::fail(GTP_E_ALIGN, "pointers must be 16-byte aligned");
  gtp::DeviceInfo dev;
  if (gtp_status s = gtp::require_sm103(&dev)) return s;
  cudaStream_t st = gtp::as_stream(stream);
  if (N == 0) return gtp::launch_zero_bytes(dX, M * K * 2, st, dev.sm_count);
  // D = dX [M, K], contraction N; A = dY [M, N] (K-major), B = W [N, K] (MN-major)
  return run_gemm<false, true, kStoreBf16>({dY, W, dX, int(M), int(K), int(N)}, false, dev, st);
}

extern "C" gtp_status gtp_linear_wgrad_accum(const void *dY, const void *X, float *grad_data, int64_t grad_offset,
                                             int64_t grad_numel_total, int64_t M, int64_t N, int64_t K, gtp_dtype dt,
                                             gtp_stream stream) {
  gtp::clear_error();
  if (dt != GTP_BF16) return gtp::fail(GTP_E_DTYPE, "only GTP_BF16 is supported");
  if (gtp_status s = check_dims(M, N, K)) return s;
  if (grad_offset < 0 || grad_numel_total < 0) return gtp::fail(GTP_E_ARG, "negative offset or size");
  if (N * K > grad_numel_total - grad_offset)
    return gtp::fail(GTP_E_RANGE, "view [%lld, +%lld) exceeds the grad buffer (%lld)", (long long)grad_offset,
                     (long long)(N * K), (long long)grad_numel_total);
  if (M == 0 || N == 0 || K == 0) return GTP_OK;
  if (!dY || !X || !grad_data) return gtp::fail(GTP_E_ARG, "null pointer");
  if (grad_offset % 4) return gtp::fail(GTP_E_ALIGN, "grad_offset must be a multiple of 4 elements");
  if (!gtp::aligned16(dY) || !gtp::aligned16(X) || !gtp::aligned16(grad_data))
    return gtp::fail(GTP_E_ALIGN, "pointers must be 16-byte aligned");
  gtp::DeviceInfo dev;
  if (gtp_status s = gtp::require_sm103(&dev)) return s;
  // D = main_grad view [N, K], contraction M; A = dY [M, N] (MN-major), B = X [M, K] (MN-major)
  return run_gemm<true, true, kReduceAddF32>({dY, X, grad_data + grad_offset, int(N), int(K), int(M)}, true, dev,
                                             gtp::as_stream(stream));
}

extern "C" gtp_status gtp_wait_timeouts(uint32_t *flags, int32_t reset) {
  gtp::clear_error();
  if (!flags) return gtp::fail(GTP_E_ARG, "null flags");
  gtp::DeviceInfo dev;
  if (gtp_status s = gtp::current_device(&dev)) return s;
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_gtp_wait_timeouts, sizeof(v));
  if (e == cudaSuccess && reset) {
    const unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_gtp_wait_timeouts, &z, sizeof(z));
  }
  if (e != cudaSuccess) return gtp::fail(GTP_E_CUDA, "reading the wait-timeout word: %s", cudaGetErrorString(e));
  *flags = v;
  return GTP_OK;
}

namespace {

// D[m_dim, n_dim] (bf16 store, or fp32 reduce-add) = dq(Aq, As) dq(Bq, Bs)^T, both operands
// K-major code rows of k_dim elements (E4M3 bytes, or packed E2M1 pairs) with one scale
// byte per block (32 for MXFP8, 16 for NVFP4).
template <int FMT, int EPI, int S>
gtp_status launch_blockscaled(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &d, const uint8_t *As,
                              const uint8_t *Bs, const float *a_amax, const float *b_amax, const Problem &p, int grid,
                              const gtp::DeviceInfo &dev, cudaStream_t st) {
  using F = BlockScaled<FMT, S>;
  static std::atomic<uint64_t> configured{0};
  if (gtp_status e = configure(gemm_blockscaled_kernel<FMT, EPI, S>, F::SMEM_TOTAL, configured, dev.device)) return e;
  return gtp::launch_overlapped(gemm_blockscaled_kernel<FMT, EPI, S>, grid, kBsThreads, F::SMEM_TOTAL, st,
                                FMT == kMxfp8 ? "gemm_mxfp8" : "gemm_nvfp4", a, b, d, As, Bs, a_amax, b_amax, p);
}

template <int FMT, int EPI>
gtp_status run_blockscaled(const uint8_t *Aq, const uint8_t *As, const uint8_t *Bq, const uint8_t *Bs,
                           const float *a_amax, const float *b_amax, void *D, int64_t m_dim, int64_t n_dim,
                           int64_t k_dim, bool allow_split, const gtp::DeviceInfo &dev, cudaStream_t st) {
  using F = BlockScaled<FMT>;
  CUtensorMap a, b, d;
  constexpr CU kU8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const int64_t row_bytes = FMT == kMxfp8 ? k_dim : k_dim / 2;
  if (gtp_status s = gtp::encode_tmap_2d(&a, kU8, Aq, row_bytes, m_dim, row_bytes, F::BK, BM, kSW128)) return s;
  if (gtp_status s = gtp::encode_tmap_2d(&b, kU8, Bq, row_bytes, n_dim, row_bytes, F::BK, BN, kSW128)) return s;
  // output boxes of 32 rows x 64 bytes, matching the epilogue's staging under the 64-byte swizzle
  constexpr CUtensorMapSwizzle kSW64 = CU_TENSOR_MAP_SWIZZLE_64B;
  gtp_status s = EPI == kStoreBf16
                     ? gtp::encode_tmap_2d(&d, kBF16, D, n_dim, m_dim, n_dim * 2, 32, 32, kSW64)
                     : gtp::encode_tmap_2d(&d, kF32, D, n_dim, m_dim, n_dim * 4, 16, 32, kSW64);
  if (s) return s;
  Problem p;
  p.m_dim = int(m_dim);
  p.n_dim = int(n_dim);
  p.k_dim = int(k_dim);
  p.tiles_m = int((m_dim + BM - 1) / BM);
  p.tiles_n = int((n_dim + BN - 1) / BN);
  p.k_blocks = int(k_dim / F::K_STAGE);
  const int tiles = p.tiles_m * p.tiles_n;
  p.splits = allow_split ? choose_splits(tiles, p.k_blocks, dev.sm_count) : 1;
  p.num_units = tiles * p.splits;
  p.group_m = 16;
  const int grid = std::min(p.num_units, dev.sm_count);
  // measured on the fc1 shape: 4 stages gain on K = 2048 (16 k-blocks per tile), 3 gain on
  // K = 8192 (64 per tile)
  if constexpr (FMT == kMxfp8)
    if (p.k_blocks / p.splits <= 16)
      return launch_blockscaled<FMT, EPI, 4>(a, b, d, As, Bs, a_amax, b_amax, p, grid, dev, st);
  return launch_blockscaled<FMT, EPI, 3>(a, b, d, As, Bs, a_amax, b_amax, p, grid, dev, st);
}

template <int EPI>
gtp_status run_mxfp8(const uint8_t *Aq, const uint8_t *As, const uint8_t *Bq, const uint8_t *Bs, void *D, int64_t m_dim,
                     int64_t n_dim, int64_t k_dim, bool allow_split, const gtp::DeviceInfo &dev, cudaStream_t st) {
  return run_blockscaled<kMxfp8, EPI>(Aq, As, Bq, Bs, nullptr, nullptr, D, m_dim, n_dim, k_dim, allow_split, dev, st);
}

// Checks shared by the MXFP8 entry points: D has m_dim x n_dim elements of `out_bytes`, the
// contraction is k_dim.
gtp_status check_mxfp8(const uint8_t *Aq, const uint8_t *As, const uint8_t *Bq, const uint8_t *Bs, const void *D,
                       int64_t m_dim, int64_t n_dim, int64_t k_dim, int out_bytes, int64_t k_multiple = 128) {
  if (m_dim < 0 || n_dim < 0 || k_dim < 0) return gtp::fail(GTP_E_ARG, "negative dimension");
  if (m_dim > kMaxDim || n_dim > kMaxDim || k_dim > kMaxDim) return gtp::fail(GTP_E_SHAPE, "dimension above 2^30");
  if (k_dim % k_multiple)
    return gtp::fail(GTP_E_SHAPE, "the contraction must be a multiple of %lld (whole stages of scale words)",
                     (long long)k_multiple);
  if ((n_dim * out_bytes) % 16) return gtp::fail(GTP_E_ALIGN, "output rows must be multiples of 16 bytes");
  if (m_dim == 0 || n_dim == 0) return GTP_OK;
  if (!D || (k_dim > 0 && (!Aq || !As || !Bq || !Bs))) return gtp::fail(GTP_E_ARG, "null pointer");
  if (!gtp::aligned16(D) || (k_dim > 0 && (!gtp::aligned16(Aq) || !gtp::aligned16(Bq))))
    return gtp::fail(GTP_E_ALIGN, "output and code pointers must be 16-byte aligned");
  // scale words are gathered with 4-byte loads: a weight's scale view inside a native
  // MXFP8 buffer starts at offset / 32, a multiple of 4 bytes for 128-aligned offsets
  if (k_dim > 0 && ((reinterpret_cast<uintptr_t>(As) | reinterpret_cast<uintptr_t>(Bs)) & 3u))
    return gtp::fail(GTP_E_ALIGN, "scale pointers must be 4-byte aligned");
  return GTP_OK;
}

}  // namespace

extern "C" gtp_status gtp_linear_fprop_mxfp8(const uint8_t *Xq, const uint8_t *Xs, const uint8_t *Wq,
                                             const uint8_t *Ws, void *Y, int64_t M, int64_t N, int64_t K,
                                             gtp_stream stream) {
  gtp::clear_error();
  if (gtp_status s = check_mxfp8(Xq, Xs, Wq, Ws, Y, M, N, K, 2)) return s;
  if (M == 0 || N == 0) return GTP_OK;
  gtp::DeviceInfo dev;
  if (gtp_status s = gtp::require_sm103(&dev)) return s;
  cudaStream_t st = gtp::as_stream(stream);
  if (K == 0) return gtp::launch_zero_bytes(Y, M * N * 2, st, dev.sm_count);
  return run_mxfp8<kStoreBf16>(Xq, Xs, Wq, Ws, Y, M, N, K, false, dev, st);
}

extern "C" gtp_status gtp_linear_dgrad_mxfp8(const uint8_t *dYq, const uint8_t *dYs, const uint8_t *Wtq,
                                             const uint8_t *Wts, void *dX, int64_t M, int64_t N, int64_t K,
                                             gtp_stream stream) {
  gtp::clear_error();
  // dX[M, K] = dq(dYq)[M, N] · dq(Wtq)[K, N]^T: contraction N, output columns K
  if (gtp_status s = check_mxfp8(dYq, dYs, Wtq, Wts, dX, M, K, N, 2)) return s;
  if (M == 0 || K == 0) return GTP_OK;
  gtp::DeviceInfo dev;
  if (gtp_status s = gtp::require_sm103(&dev)) return s;
  cudaStream_t st = gtp::as_stream(stream);
  if (N == 0) return gtp::launch_zero_bytes(dX, M * K * 2, st, dev.sm_count);
  return run_mxfp8<kStoreBf16>(dYq, dYs, Wtq, Wts, dX, M, K, N, false, dev, st);
}

extern "C" gtp_status gtp_linear_wgrad_accum_mxfp8(const uint8_t *dYtq, const uint8_t *dYts, const uint8_t *Xtq,
                                                   const uint8_t *Xts, float *grad_data, int64_t grad_offset,
                                                   int64_t grad_numel_total, int64_t M, int64_t N, int64_t K,
                                                   gtp_stream stream) {
  gtp::clear_error();
  // main_grad[N, K] += dq(dYtq)[N, M] · dq(Xtq)[K, M]^T: contraction M
  if (grad_offset < 0 || grad_numel_total < 0) return gtp::fail(GTP_E_ARG, "negative offset or size");
  if (N * K > grad_numel_total - grad_offset)
    return gtp::fail(GTP_E_RANGE, "view [%lld, +%lld) exceeds the grad buffer (%lld)", (long long)grad_offset,
                     (long long)(N * K), (long long)grad_numel_total);
  if (grad_offset % 4) return gtp::fail(GTP_E_ALIGN, "grad_offset must be a multiple of 4 elements");
  float *view = grad_data ? grad_data + grad_offset : nullptr;
  if (gtp_status s = check_mxfp8(dYtq, dYts, Xtq, Xts, view, N, K, M, 4)) return s;
  if (M == 0 || N == 0 || K == 0) return GTP_OK;
  gtp::DeviceInfo dev;
  if (gtp_status s = gtp::require_sm103(&dev)) return s;
  return run_mxfp8<kReduceAddF32>(dYtq, dYts, Xtq, Xts, view, N, K, M, true, dev, gtp::as_stream(stream));
}

extern "C" gtp_status gtp_linear_fprop_nvfp4(const uint8_t *Xq, const uint8_t *Xs, const float *x_amax,
                                             const uint8_t *Wq, const uint8_t *Ws, const float *w_amax, void *Y,
                                             int64_t M, int64_t N, int64_t K, gtp_stream stream) {
  gtp::clear_error();
  if (gtp_status s = check_mxfp8(Xq, Xs, Wq, Ws, Y, M, N, K, 2, BlockScaled<kNvfp4>::K_STAGE)) return s;
  if (M == 0 || N == 0) return GTP_OK;
  if (K > 0 && (!x_amax || !w_amax)) return gtp::fail(GTP_E_ARG, "null amax");
  if ((reinterpret_cast<uintptr_t>(x_amax) | reinterpret_cast<uintptr_t>(w_amax)) & 3u)
    return gtp::fail(GTP_E_ALIGN, "amax pointers must be 4-byte aligned");
  // a stage's four scale words of a row are one 16-byte load
  if (K > 0 && (!gtp::aligned16(Xs) || !gtp::aligned16(Ws)))
    return gtp::fail(GTP_E_ALIGN, "NVFP4 scale pointers must be 16-byte aligned");
  gtp::DeviceInfo dev;
  if (gtp_status s = gtp::require_sm103(&dev)) return s;
  cudaStream_t st = gtp::as_stream(stream);
  if (K == 0) return gtp::launch_zero_bytes(Y, M * N * 2, st, dev.sm_count);
  return run_blockscaled<kNvfp4, kStoreBf16>(Xq, Xs, Wq, Ws, x_amax, w_amax, Y, M, N, K, false, dev, st);
}
