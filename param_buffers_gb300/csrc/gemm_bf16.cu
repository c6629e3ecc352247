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
#include <map>
#include <type_traits>
#include <mutex>
#include <vector>

#include "gemm_common.cuh"

namespace gtp {
// The wait-timeout word of the block-scaled unit (gemm_blockscaled.cu).
gtp_status blockscaled_wait_word(unsigned int *v, bool reset);
}

namespace {

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
  } else if (warp == 1) {  // -------------- MMA issuer: the whole warp waits, one elected lane issues
    const uint32_t idesc = idesc_bf16_f32(BM, BN, A_MN, B_MN);
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
      int tm, tn, kb0, kb1;
      decode_unit(p, u, tm, tn, kb0, kb1);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, err, 0x2u))) break;
      tc_fence_after();
      const uint32_t d = tmem_base + uint32_t(acc * BN);
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[stage], phase, abort_flag, err, 0x4u))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (elect_one_sync()) {
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
        }
        __syncwarp();
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (elect_one_sync()) mma_commit(&tfull[acc]);
      __syncwarp();
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (elect_one_sync()) mma_commit(drain);  // every issued MMA has finished before tensor memory is freed
    __syncwarp();
    if (lane == 0) drain_wait(drain, 0);
  } else {  // -------------------------------------------------------------- epilogue
    const int ew = warp - 2;
    const int quarter = warp & 3;  // tensor-memory lanes 32*quarter .. +31 belong to this warp
    uint8_t *mybuf = sEpi + ew * 2 * EPI_BUF;
    int acc = 0, bufsel = 0;
    uint32_t acc_phase = 0;
    constexpr int CW = (EPI == kStoreBf16 || EPI == kAccumBf16) ? 64 : 32;  // columns per 128-byte row
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
        if (CW == 64) tmem_ld_32x32b_x32(tbase + uint32_t(c * CW + 32), r1);
        tmem_ld_wait();
        if constexpr (EPI == kReduceAddF32Direct) {
          red_row_f32(p.direct, row + lane, tn * BN + c * CW, p.m_dim, p.n_dim, r0);
          continue;
        } else if constexpr (EPI == kAccumBf16) {
          accum_row_bf16(p.direct, row + lane, tn * BN + c * CW, p.m_dim, p.n_dim, r0, r1);
          continue;
        }
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
//   In each CTA, warp 0 issues the A copies and warp 6 the B copies of every stage.  Both
//   CTAs' TMA copies complete on the even CTA's full[] barrier (cta_group::2 loads),
//   which the even CTA's warp 0 arms for the bytes of both halves; its warp 1 issues the MMAs and
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
// warps: 0 A producer (arms each stage), 1 MMA, 2-5 epilogue, 6 B producer
constexpr int kThreads = kGemmThreads + 32;
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
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(pair::kThreads, 1)
    gemm_bf16_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmBh, const __grid_constant__ CUtensorMap tmD,
                          const Problem p) {
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
    tma_prefetch_desc(&tmBh);
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
      const uint64_t pol_a = l2_policy(p.hint_a), pol_b = l2_policy(p.hint_b);
      if (DYN && unit >= 0 && !clc_request(rank == 0, slot, sphase, resp, clc_full, clc_empty, abort_flag, err))
        unit = -1;
      while (unit >= 0) {
        int tm, tn, kb0, kb1, half;
        decode_unit_half(p, unit, tm, tn, kb0, kb1, half);
        const int m0 = tm * pair::BMP + pair::BMC * int(rank);
        // a half-width unit takes 64 B rows a CTA (a 64-row box, or one 64-wide MN chunk)
        const int n0 = tn * BN + (half < 0 ? pair::BNC * int(rank) : (BN / 2) * half + (pair::BNC / 2) * int(rank));
        const uint32_t stage_tx = 2u * uint32_t(half < 0 ? pair::STAGE_BYTES : pair::A_STAGE + pair::B_STAGE / 2);
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, err, 0x1u)) {
            ok = false;
            break;
          }
          if (rank == 0) {  // the even CTA's barrier counts both CTAs' bytes
            mbar_arrive_expect_tx(&full[stage], stage_tx);
            armed[stage] = int(phase);
          }
          const uint32_t bar = mapa_shared(&full[stage], 0);
          uint8_t *a = sA + stage * pair::A_STAGE;
          uint8_t *b = sB + stage * pair::B_STAGE;
          const int k0 = kb * BK;
          if (A_MN) {
            tma_load_2d_pair_hint(&tmA, bar, a, m0, k0, pol_a);
            tma_load_2d_pair_hint(&tmA, bar, a + MN_CHUNK, m0 + 64, k0, pol_a);
          } else {
            tma_load_2d_pair_hint(&tmA, bar, a, k0, m0, pol_a);
          }
          if (DYN) {  // the dynamic schedule keeps one producer thread
            if (B_MN) {
              tma_load_2d_pair_hint(&tmB, bar, b, n0, k0, pol_b);
              if (half < 0) tma_load_2d_pair_hint(&tmB, bar, b + MN_CHUNK, n0 + 64, k0, pol_b);
            } else {
              tma_load_2d_pair_hint(half < 0 ? &tmB : &tmBh, bar, b, k0, n0, pol_b);
            }
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
  } else if (warp == 1) {  // -- MMA issuer (even CTA; the odd CTA only follows the units): the whole warp
    //                           waits, one elected lane issues, lane 0 advances the schedule
    int stage = 0, acc = 0, slot = 0;
    uint32_t phase = 0, acc_phase = 0, sphase = 0;
    int unit = first;
    while (unit >= 0) {
      if (rank == 0) {
        int tm, tn, kb0, kb1, half;
        decode_unit_half(p, unit, tm, tn, kb0, kb1, half);
        const uint32_t idesc = idesc_bf16_f32(pair::BMP, half < 0 ? BN : BN / 2, A_MN, B_MN);
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, err, 0x2u))) break;
        tc_fence_after();
        const uint32_t d = tmem_base + uint32_t(acc * BN);
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[stage], phase, abort_flag, err, 0x4u))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one_sync()) {
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
          }
          __syncwarp();
          if (++stage == pair::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (elect_one_sync()) mma_commit_pair(&tfull[acc], 0x3);
        __syncwarp();
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // the dynamic schedule's ring (one release a role) stays with lane 0
      int next = -1;
      if (lane == 0)
        next = advance_unit<DYN>(unit, slot, sphase, nclusters, p, resp, clc_full, clc_empty, abort_flag, err);
      unit = __shfl_sync(0xFFFFFFFFu, next, 0);
    }
    if (rank == 0) {
      if (elect_one_sync()) mma_commit_pair(drain, 0x3);  // both CTAs learn when every MMA has finished
      __syncwarp();
    }
    if (lane == 0) drain_wait(drain, 0);
  } else if (warp == 6) {
    // ------------------------------------------- B producer (both CTAs; static schedule)
    // Two threads in two warps issue a stage's copies: with 3-4 copies a stage (MN-major
    // operands) one thread's issue loop fell behind the MMAs (measured: fc1 wgrad 163.5 ->
    // 155.1 us, the O projection's unsplit wgrad 40.6 -> 33.4 us, dgrad 1-2 % faster).  B's
    // bytes may land on the even CTA's full barrier before warp 0 arms it; the phase cannot
    // complete before that arrival.
    if (!DYN && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      const uint64_t pol_b = l2_policy(p.hint_b);
      for (int unit = first; unit >= 0 && unit < p.num_units; unit += nclusters) {
        int tm, tn, kb0, kb1, half;
        decode_unit_half(p, unit, tm, tn, kb0, kb1, half);
        const int n0 = tn * BN + (half < 0 ? pair::BNC * int(rank) : (BN / 2) * half + (pair::BNC / 2) * int(rank));
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, err, 0x1u)) {
            ok = false;
            break;
          }
          const uint32_t bar = mapa_shared(&full[stage], 0);
          uint8_t *b = sB + stage * pair::B_STAGE;
          const int k0 = kb * BK;
          if (B_MN) {
            tma_load_2d_pair_hint(&tmB, bar, b, n0, k0, pol_b);
            if (half < 0) tma_load_2d_pair_hint(&tmB, bar, b + MN_CHUNK, n0 + 64, k0, pol_b);
          } else {
            tma_load_2d_pair_hint(half < 0 ? &tmB : &tmBh, bar, b, k0, n0, pol_b);
          }
          if (++stage == pair::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
    }
  } else {  // -------------------------------------------------------- epilogue (both CTAs)
    const int ew = warp - 2;
    const int quarter = warp & 3;
    uint8_t *mybuf = sEpi + ew * 2 * EPI_BUF;
    int acc = 0, bufsel = 0, slot = 0;
    uint32_t acc_phase = 0, sphase = 0;
    constexpr int CW = (EPI == kStoreBf16 || EPI == kAccumBf16) ? 64 : 32;
    int unit = first;
    while (unit >= 0) {
      int tm, tn, kb0, kb1, half;
      decode_unit_half(p, unit, tm, tn, kb0, kb1, half);
      const int ncols = half < 0 ? BN : BN / 2;
      const int col0 = tn * BN + (half < 0 ? 0 : (BN / 2) * half);
      const bool ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, err, 0x8u);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;  // the warp leaves together
      tc_fence_after();
      const int row = tm * pair::BMP + pair::BMC * int(rank) + 32 * quarter;
      const uint32_t tbase = tmem_base + (uint32_t(32 * quarter) << 16) + uint32_t(acc * BN);
#pragma unroll 1
      for (int c = 0; c < ncols / CW; ++c) {
        uint32_t r0[32], r1[32];
        tmem_ld_32x32b_x32(tbase + uint32_t(c * CW), r0);
        if (CW == 64) tmem_ld_32x32b_x32(tbase + uint32_t(c * CW + 32), r1);
        tmem_ld_wait();
        if constexpr (EPI == kReduceAddF32Direct) {
          red_row_f32(p.direct, row + lane, col0 + c * CW, p.m_dim, p.n_dim, r0);
          continue;
        } else if constexpr (EPI == kAccumBf16) {
          accum_row_bf16(p.direct, row + lane, col0 + c * CW, p.m_dim, p.n_dim, r0, r1);
          continue;
        }
        uint8_t *buf = mybuf + bufsel * EPI_BUF;
        if (lane == 0) bulk_wait_group_read<1>();
        __syncwarp();
        stage_rows<EPI>(buf, lane, r0, r1);
        fence_proxy_async_smem();
        __syncwarp();
        const int col = col0 + c * CW;
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
      // every load of the accumulator has completed (wait::ld); a release would also wait for
      // the stores just issued
      if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(&tempty[acc], 0));
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

// --------------------------------------------------------------------------- grouped CTA-pair GEMM
//
// Several independent products in ONE persistent launch of the CTA-pair kernel: a linear's
// dgrad and wgrad (both read dY, neither needs the other: [LIN] §4.2 computes them in the
// same backward), or any list of up to kMaxItems fprop / dgrad / wgrad products.  The
// units (tile, contraction range) of all products form one list, product after product,
// that the pairs take round-robin, so the start-up, the last wave and the last epilogue
// are paid once for the whole group, and one product's short last wave is filled with
// another's units.  Operand majorness and the epilogue (bf16 store, fp32 reduce-add, or
// one of the register epilogues) are per product; everything else is the CTA-pair kernel
// above.
//
// Each role runs a unit through a function templated on the product's index, so every
// parameter read and every tensor-map address is a compile-time offset into the kernel
// parameter.  Read with a run-time index, the fields became generic loads that every
// tensor instruction's memory clobber forced the compiler to repeat, and the tensor-map
// address of each copy had to be made warp-uniform at run time: the producer then fell
// behind the MMAs (measured 580-750 cycles a stage against 512).
namespace grp {
constexpr int kMaxItems = 4;
struct Item {
  Problem p;             // shape, tiles, splits, half-width tail, L2 policies
  int32_t a_mn, b_mn;    // operand majorness: 0 K-major, 1 MN-major
  int32_t epi;           // kStoreBf16 or kReduceAddF32
  int32_t unit_begin;    // first unit of this product in the group's unit list
};
struct Maps {
  CUtensorMap a, b, bh, d;
};
struct Args {
  Maps maps[kMaxItems];
  Item it[kMaxItems];
  int32_t n, num_units;
};
}  // namespace grp

__device__ __forceinline__ int group_item(const grp::Args &g, int u) {
  int i = 0;
#pragma unroll
  for (int j = 1; j < grp::kMaxItems; ++j)  // constant indices: plain parameter reads
    if (j < g.n && u >= g.it[j].unit_begin) i = j;
  return i;
}

// Calls f(std::integral_constant<int, i>) for the run-time product index i.
template <typename F>
__device__ __forceinline__ void with_item(int i, F &&f) {
  static_assert(grp::kMaxItems == 4, "one case per product");
  switch (i) {
    case 0: f(std::integral_constant<int, 0>()); break;
    case 1: f(std::integral_constant<int, 1>()); break;
    case 2: f(std::integral_constant<int, 2>()); break;
    default: f(std::integral_constant<int, 3>()); break;
  }
}

// Shared-memory ring state of the producer and the MMA issuer.
struct Ring {
  int stage = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next() {
    if (++stage == pair::STAGES) {
      stage = 0;
      phase ^= 1u;
    }
  }
};

// TMA producer, one unit of product I (both CTAs), with the operand majorness fixed at
// compile time so that the stage loop holds no branch on it.  Returns false when a wait
// gave up.
template <int I, bool A_MN, bool B_MN, int PART>
__device__ __forceinline__ bool group_produce_t(const grp::Args &g, int local_unit, uint32_t rank, Ring &ring,
                                                int *armed, uint8_t *sA, uint8_t *sB, uint64_t *full,
                                                uint64_t *empty, uint64_t pol_a, uint64_t pol_b,
                                                volatile int *abort_flag, unsigned int *err) {
  int tm, tn, kb0, kb1, half;
  decode_unit_half(g.it[I].p, local_unit, tm, tn, kb0, kb1, half);
  const int m0 = tm * pair::BMP + pair::BMC * int(rank);
  const int n0 = tn * BN + (half < 0 ? pair::BNC * int(rank) : (BN / 2) * half + (pair::BNC / 2) * int(rank));
  const uint32_t stage_tx = 2u * uint32_t(half < 0 ? pair::STAGE_BYTES : pair::A_STAGE + pair::B_STAGE / 2);
  const CUtensorMap *mb = (B_MN || half < 0) ? &g.maps[I].b : &g.maps[I].bh;
  for (int kb = kb0; kb < kb1; ++kb) {
    if (!mbar_wait(&empty[ring.stage], ring.phase ^ 1u, abort_flag, err, 0x1u)) return false;
    const uint32_t bar = mapa_shared(&full[ring.stage], 0);
    const int k0 = kb * BK;
    if (PART == 0) {  // A, and the stage's arming
      if (rank == 0) {  // the even CTA's barrier counts both CTAs' bytes
        mbar_arrive_expect_tx(&full[ring.stage], stage_tx);
        armed[ring.stage] = int(ring.phase);
      }
      uint8_t *a = sA + ring.stage * pair::A_STAGE;
      if (A_MN) {
        tma_load_2d_pair_hint(&g.maps[I].a, bar, a, m0, k0, pol_a);
        tma_load_2d_pair_hint(&g.maps[I].a, bar, a + MN_CHUNK, m0 + 64, k0, pol_a);
      } else {
        tma_load_2d_pair_hint(&g.maps[I].a, bar, a, k0, m0, pol_a);
      }
    } else {  // B
      uint8_t *b = sB + ring.stage * pair::B_STAGE;
      if (B_MN) {
        tma_load_2d_pair_hint(mb, bar, b, n0, k0, pol_b);
        if (half < 0) tma_load_2d_pair_hint(mb, bar, b + MN_CHUNK, n0 + 64, k0, pol_b);
      } else {
        tma_load_2d_pair_hint(mb, bar, b, k0, n0, pol_b);
      }
    }
    ring.next();
  }
  return true;
}

// PART 0: warp 0 issues A's copies and arms each stage; PART 1: warp 6 issues B's.
template <int I, int PART>
__device__ __forceinline__ bool group_produce(const grp::Args &g, int local_unit, uint32_t rank, Ring &ring,
                                              int *armed, uint8_t *sA, uint8_t *sB, uint64_t *full,
                                              uint64_t *empty, const uint64_t (&pol)[3], volatile int *abort_flag,
                                              unsigned int *err) {
  const grp::Item &it = g.it[I];
  const uint64_t pa = pol[it.p.hint_a], pb = pol[it.p.hint_b];
  if (PART == 0)
    return it.a_mn ? group_produce_t<I, true, false, 0>(g, local_unit, rank, ring, armed, sA, sB, full, empty, pa,
                                                        pb, abort_flag, err)
                   : group_produce_t<I, false, false, 0>(g, local_unit, rank, ring, armed, sA, sB, full, empty, pa,
                                                         pb, abort_flag, err);
  return it.b_mn ? group_produce_t<I, false, true, 1>(g, local_unit, rank, ring, armed, sA, sB, full, empty, pa, pb,
                                                      abort_flag, err)
                 : group_produce_t<I, false, false, 1>(g, local_unit, rank, ring, armed, sA, sB, full, empty, pa, pb,
                                                       abort_flag, err);
}

// MMA issuer, one unit of product I (even CTA; the whole warp waits, one elected lane
// issues).  Returns false when a wait gave up.
template <int I>
__device__ __forceinline__ bool group_mma(const grp::Args &g, int local_unit, Ring &ring, uint32_t d,
                                          uint8_t *sA, uint8_t *sB, uint64_t *full, uint64_t *empty,
                                          volatile int *abort_flag, unsigned int *err) {
  const grp::Item &it = g.it[I];
  int tm, tn, kb0, kb1, half;
  decode_unit_half(it.p, local_unit, tm, tn, kb0, kb1, half);
  const bool a_mn = it.a_mn != 0, b_mn = it.b_mn != 0;
  const uint32_t idesc = idesc_bf16_f32(pair::BMP, half < 0 ? BN : BN / 2, a_mn, b_mn);
  // per-k step of the descriptors' start address and their leading-byte offset
  const uint32_t a_step = a_mn ? UK * 128 : UK * 2, b_step = b_mn ? UK * 128 : UK * 2;
  const uint32_t a_lbo = a_mn ? MN_CHUNK : 16, b_lbo = b_mn ? MN_CHUNK : 16;
  for (int kb = kb0; kb < kb1; ++kb) {
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[ring.stage], ring.phase, abort_flag, err, 0x4u))) return false;
    tc_fence_after();
    if (elect_one_sync()) {
      const uint32_t a0 = smem_u32(sA + ring.stage * pair::A_STAGE);
      const uint32_t b0 = smem_u32(sB + ring.stage * pair::B_STAGE);
#pragma unroll
      for (int k = 0; k < BK / UK; ++k)
        mma_f16_pair(d, sdesc_sw128(a0 + k * a_step, a_lbo, 1024), sdesc_sw128(b0 + k * b_step, b_lbo, 1024), idesc,
                     (kb > kb0 || k > 0) ? 1u : 0u);
      mma_commit_pair(&empty[ring.stage], 0x3);
    }
    __syncwarp();
    ring.next();
  }
  return true;
}

// The epilogue of one accumulator tile: `ncols` columns of this warp's 32 rows, converted
// (bf16) or not (fp32) and sent by TMA as a store or a reduce-add, or added by the
// register epilogues straight into `direct` (fp32 atomics, or the bf16 read-add-write).
template <int EPI>
__device__ __forceinline__ void group_epilogue(const CUtensorMap *tmD, void *direct, uint32_t tbase, int ncols,
                                               int row, int col0, int m_dim, int n_dim, uint8_t *mybuf, int &bufsel,
                                               int lane) {
  constexpr int CW = (EPI == kStoreBf16 || EPI == kAccumBf16) ? 64 : 32;
#pragma unroll 1
  for (int c = 0; c < ncols / CW; ++c) {
    uint32_t r0[32], r1[32];
    tmem_ld_32x32b_x32(tbase + uint32_t(c * CW), r0);
    if (CW == 64) tmem_ld_32x32b_x32(tbase + uint32_t(c * CW + 32), r1);
    tmem_ld_wait();
    if constexpr (EPI == kReduceAddF32Direct) {
      red_row_f32(direct, row + lane, col0 + c * CW, m_dim, n_dim, r0);
      continue;
    } else if constexpr (EPI == kAccumBf16) {
      accum_row_bf16(direct, row + lane, col0 + c * CW, m_dim, n_dim, r0, r1);
      continue;
    }
    uint8_t *buf = mybuf + bufsel * EPI_BUF;
    if (lane == 0) bulk_wait_group_read<1>();
    __syncwarp();
    stage_rows<EPI>(buf, lane, r0, r1);
    fence_proxy_async_smem();
    __syncwarp();
    const int col = col0 + c * CW;
    if (lane == 0) {
      if (row < m_dim && col < n_dim) {
        if (EPI == kStoreBf16)
          tma_store_2d(tmD, buf, col, row);
        else
          tma_reduce_add_2d(tmD, buf, col, row);
      }
      bulk_commit_group();
    }
    bufsel ^= 1;
  }
}

// Epilogue warp, one unit of product I.
template <int I>
__device__ __forceinline__ void group_store(const grp::Args &g, int local_unit, uint32_t rank, int quarter,
                                            uint32_t tbase, uint8_t *mybuf, int &bufsel, int lane) {
  const grp::Item &it = g.it[I];
  int tm, tn, kb0, kb1, half;
  decode_unit_half(it.p, local_unit, tm, tn, kb0, kb1, half);
  const int ncols = half < 0 ? BN : BN / 2;
  const int col0 = tn * BN + (half < 0 ? 0 : (BN / 2) * half);
  const int row = tm * pair::BMP + pair::BMC * int(rank) + 32 * quarter;
  const CUtensorMap *tmD = &g.maps[I].d;
  switch (it.epi) {
    case kStoreBf16:
      group_epilogue<kStoreBf16>(tmD, it.p.direct, tbase, ncols, row, col0, it.p.m_dim, it.p.n_dim, mybuf, bufsel,
                                 lane);
      break;
    case kReduceAddF32:
      group_epilogue<kReduceAddF32>(tmD, it.p.direct, tbase, ncols, row, col0, it.p.m_dim, it.p.n_dim, mybuf, bufsel,
                                    lane);
      break;
    case kReduceAddF32Direct:
      group_epilogue<kReduceAddF32Direct>(tmD, it.p.direct, tbase, ncols, row, col0, it.p.m_dim, it.p.n_dim, mybuf,
                                          bufsel, lane);
      break;
    default:
      group_epilogue<kAccumBf16>(tmD, it.p.direct, tbase, ncols, row, col0, it.p.m_dim, it.p.n_dim, mybuf, bufsel,
                                 lane);
      break;
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(pair::kThreads, 1)
    gemm_bf16_group_kernel(const __grid_constant__ grp::Args g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + pair::STAGES * pair::A_STAGE;
  uint8_t *sEpi = smem + pair::SMEM_OPS;
  uint64_t *full = reinterpret_cast<uint64_t *>(sEpi + SMEM_EPI);
  uint64_t *empty = full + pair::STAGES;
  uint64_t *tfull = empty + pair::STAGES;
  uint64_t *tempty = tfull + 2;
  uint64_t *drain = tempty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
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
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane < g.n)
    with_item(lane, [&](auto I) {
      tma_prefetch_desc(&g.maps[I.value].a);
      tma_prefetch_desc(&g.maps[I.value].b);
      tma_prefetch_desc(&g.maps[I.value].bh);
      tma_prefetch_desc(&g.maps[I.value].d);
    });
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
  allow_dependents();
  wait_prior_grid();

  if (warp == 0) {
    if (lane == 0) {  // ------------------------------------------ TMA producer (both CTAs)
      Ring ring;
      int armed[pair::STAGES];
      for (int s = 0; s < pair::STAGES; ++s) armed[s] = -1;
      const uint64_t pol[3] = {l2_policy(0), l2_policy(1), l2_policy(2)};
      for (int unit = cluster; unit < g.num_units; unit += nclusters) {
        const int i = group_item(g, unit);
        bool ok = true;
        with_item(i, [&](auto I) {
          ok = group_produce<I.value, 0>(g, unit - g.it[I.value].unit_begin, rank, ring, armed, sA, sB, full, empty,
                                         pol, abort_flag, err);
        });
        if (!ok) break;
      }
      for (int s = 0; s < pair::STAGES; ++s)
        if (armed[s] >= 0) drain_wait(&full[s], uint32_t(armed[s]));
    }
  } else if (warp == 1) {  // -------------------------------- MMA issuer (even CTA; the whole warp waits)
    if (rank == 0) {
      Ring ring;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int unit = cluster; unit < g.num_units; unit += nclusters) {
        const int i = group_item(g, unit);
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, err, 0x2u))) break;
        tc_fence_after();
        const uint32_t d = tmem_base + uint32_t(acc * BN);
        bool ok = true;
        with_item(i, [&](auto I) {
          ok = group_mma<I.value>(g, unit - g.it[I.value].unit_begin, ring, d, sA, sB, full, empty, abort_flag, err);
        });
        if (!ok) break;
        if (elect_one_sync()) mma_commit_pair(&tfull[acc], 0x3);
        __syncwarp();
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (elect_one_sync()) mma_commit_pair(drain, 0x3);  // both CTAs learn when every MMA has finished
      __syncwarp();
    }
    if (lane == 0) drain_wait(drain, 0);
  } else if (warp == 6) {  // ------------------------------------------- B producer (both CTAs)
    if (lane == 0) {
      Ring ring;
      const uint64_t pol[3] = {l2_policy(0), l2_policy(1), l2_policy(2)};
      for (int unit = cluster; unit < g.num_units; unit += nclusters) {
        const int i = group_item(g, unit);
        bool ok = true;
        with_item(i, [&](auto I) {
          ok = group_produce<I.value, 1>(g, unit - g.it[I.value].unit_begin, rank, ring, nullptr, sA, sB, full,
                                         empty, pol, abort_flag, err);
        });
        if (!ok) break;
      }
    }
  } else {  // -------------------------------------------------------- epilogue (both CTAs)
    const int ew = warp - 2;
    const int quarter = warp & 3;
    uint8_t *mybuf = sEpi + ew * 2 * EPI_BUF;
    int acc = 0, bufsel = 0;
    uint32_t acc_phase = 0;
    for (int unit = cluster; unit < g.num_units; unit += nclusters) {
      const int i = group_item(g, unit);
      const bool ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, err, 0x8u);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (uint32_t(32 * quarter) << 16) + uint32_t(acc * BN);
      with_item(i, [&](auto I) {
        group_store<I.value>(g, unit - g.it[I.value].unit_begin, rank, quarter, tbase, mybuf, bufsel, lane);
      });
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(&tempty[acc], 0));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
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

// --------------------------------------------------------------------------- host side

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

// Co-resident CTA pairs of the pair kernel on the current device (cached per device).
template <typename K>
int max_pairs(K kernel, const gtp::DeviceInfo &dev) {
  static std::atomic<int> cached[64];
  int v = cached[dev.device & 63].load();
  if (v > 0) return v;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(dev.sm_count & ~1));
  cfg.blockDim = dim3(pair::kThreads);
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

// The four tensor maps of a product: A and B operands (boxes of one stage, as the
// kernel's majorness reads them), B again with half the rows for half-width tail units
// (K-major B on the CTA pair), and D (the bf16 output or the fp32 main_grad view).
gtp_status encode_maps(const Operands &o, bool a_mn, bool b_mn, int epi, bool pr, CUtensorMap &ta, CUtensorMap &tb,
                       CUtensorMap &tbh, CUtensorMap &td) {
  const uint32_t b_rows = pr ? pair::BNC : BN;  // B rows staged per CTA
  gtp_status s;
  if (a_mn)
    s = gtp::encode_tmap_2d(&ta, kBF16, o.a, o.m_dim, o.k_dim, uint64_t(o.m_dim) * 2, 64, BK, kSW128);
  else
    s = gtp::encode_tmap_2d(&ta, kBF16, o.a, o.k_dim, o.m_dim, uint64_t(o.k_dim) * 2, 64, BM, kSW128);
  if (s) return s;
  if (b_mn)
    s = gtp::encode_tmap_2d(&tb, kBF16, o.b, o.n_dim, o.k_dim, uint64_t(o.n_dim) * 2, 64, BK, kSW128);
  else
    s = gtp::encode_tmap_2d(&tb, kBF16, o.b, o.k_dim, o.n_dim, uint64_t(o.k_dim) * 2, 64, b_rows, kSW128);
  if (s) return s;
  tbh = tb;  // the CTA pair's half-width tail units load 64 K-major B rows a CTA
  if (pr && !b_mn) s = gtp::encode_tmap_2d(&tbh, kBF16, o.b, o.k_dim, o.n_dim, uint64_t(o.k_dim) * 2, 64, b_rows / 2, kSW128);
  if (s) return s;
  if (epi == kStoreBf16)
    return gtp::encode_tmap_2d(&td, kBF16, o.d, o.n_dim, o.m_dim, uint64_t(o.n_dim) * 2, 64, 32, kSW128);
  if (epi == kReduceAddF32)
    return gtp::encode_tmap_2d(&td, kF32, o.d, o.n_dim, o.m_dim, uint64_t(o.n_dim) * 4, 32, 32, kSW128);
  td = tb;  // register epilogues write D themselves; the kernel only prefetches this (valid) map
  return GTP_OK;
}

// Tile counts of a product on the CTA pair (pr) or the single-CTA kernel.
Problem tile_problem(const Operands &o, bool pr) {
  const int bm = pr ? pair::BMP : BM;
  Problem p;
  p.m_dim = o.m_dim;
  p.n_dim = o.n_dim;
  p.k_dim = o.k_dim;
  p.tiles_m = (o.m_dim + bm - 1) / bm;
  p.tiles_n = (o.n_dim + BN - 1) / BN;
  p.k_blocks = (o.k_dim + BK - 1) / BK;
  return p;
}

// When the operands overflow a good part of L2, the smaller one (re-read by every wave of
// tiles) is loaded evict_last and the larger (read once per wave) evict_first.
// GTP_GEMM_L2HINT=off (read at each call) loads both with the normal policy.
void set_l2_hints(const Operands &o, Problem &p) {
  const char *hint_env = std::getenv("GTP_GEMM_L2HINT");
  const double a_bytes = 2.0 * o.m_dim * o.k_dim, b_bytes = 2.0 * o.n_dim * o.k_dim;
  constexpr double kL2Share = 48.0 * (1 << 20);  // about a third of the 126 MB L2
  if (!(hint_env && !std::strcmp(hint_env, "off")) && a_bytes + b_bytes > 2 * kL2Share &&
      std::min(a_bytes, b_bytes) <= kL2Share) {
    p.hint_a = a_bytes <= b_bytes ? 2 : 1;
    p.hint_b = a_bytes <= b_bytes ? 1 : 2;
  }
}

template <bool A_MN, bool B_MN, int EPI>
gtp_status run_gemm(const Operands &o, bool allow_split, const gtp::DeviceInfo &dev, cudaStream_t stream) {
  const bool pr = use_pair(o.m_dim);
  CUtensorMap ta, tb, tbh, td;
  if (gtp_status s = encode_maps(o, A_MN, B_MN, EPI, pr, ta, tb, tbh, td)) return s;
  Problem p = tile_problem(o, pr);
  // The CTA pair walks its tiles row by row (groups of one pair-tile row): a wave of 76
  // tiles then holds several whole rows, each row's A block is read once by all the tiles
  // that need it, and B (read by every wave) stays in L2.  Measured at the fc1 shape:
  // groups of 2 rows against groups of 8 cut the DRAM reads of dgrad from 281 to 201 MB
  // and of wgrad from 410 to 294 MB (2-4 % faster); one row at a time against groups of 2
  // then gave the layer step +0.5-0.9 %, with fc1 wgrad moving 1.04x its minimum traffic.
  p.group_m = pr ? 1 : 16;
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
    finalize_problem(p);
    // A last partial wave of T tiles with 2T <= pairs runs as 2T half-width (256 x 128)
    // units, one per pair, and takes half a tile's time.  GTP_GEMM_TAIL=full (read at each
    // call) keeps whole tiles.
    const int tail = tiles % pairs;
    const char *tail_env = std::getenv("GTP_GEMM_TAIL");
    if (!dyn && p.splits == 1 && tail > 0 && 2 * tail <= pairs && !(tail_env && !std::strcmp(tail_env, "full"))) {
      p.tail_first = tiles - tail;
      p.tail_half = 1;
      p.num_units = p.tail_first + 2 * tail;
    }
    set_l2_hints(o, p);
    p.direct = o.d;
    const int grid = 2 * (dyn ? p.num_units : std::min(p.num_units, pairs));
    return gtp::launch_overlapped(kernel, grid, pair::kThreads, pair::SMEM_TOTAL, stream, "gemm_bf16_pair_kernel", ta,
                                  tb, tbh, td, p);
  }
  static std::atomic<uint64_t> configured{0};
  auto kernel = gemm_bf16_kernel<A_MN, B_MN, EPI>;
  if (gtp_status e = configure(kernel, SMEM_TOTAL, configured, dev.device)) return e;
  p.splits = allow_split ? choose_splits(tiles, p.k_blocks, dev.sm_count) : 1;
  p.num_units = tiles * p.splits;
  finalize_problem(p);
  p.direct = o.d;
  const int grid = std::min(p.num_units, dev.sm_count);
  return gtp::launch_overlapped(kernel, grid, kGemmThreads, SMEM_TOTAL, stream, "gemm_bf16_kernel", ta, tb, td, p);
}

gtp_status check_dims(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 0) return gtp::fail(GTP_E_ARG, "negative dimension");
  if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return gtp::fail(GTP_E_SHAPE, "dimension above 2^30");
  if (N % 8 || K % 8) return gtp::fail(GTP_E_ALIGN, "N and K must be multiples of 8 (16-byte rows)");
  return GTP_OK;
}

// ------------------------------------------------------------------ grouped launch (host)

// One product of a group as the host hands it to the grouped kernel.
struct GroupSpec {
  Operands o;
  bool a_mn, b_mn;
  int epi;
  bool may_split;  // a reduce-add product whose contraction may be split across pairs
};

// Cost of a half-width (256 x 128) unit relative to a whole tile of the same contraction:
// its MMAs take half the time, but each stage still loads all 256 A rows.  Measured on the
// O-projection wgrad: 64 half-width units of 128 k-blocks took 41.0 us against 26.6 us
// for 64 whole tiles of 64 k-blocks, i.e. 0.77 of a whole tile rather than 0.5.
constexpr double kHalfUnitCost = 0.77;

// Modeled busy time, in k-blocks of a 256-wide tile, of the pair that finishes last when
// the products' units, in the order given, are taken round-robin by `pairs` CTA pairs (as
// the grouped kernel takes them); with `tail`, the last partial wave's units (all of the
// last product, which is unsplit) run as twice as many half-width units.
double group_makespan(const std::vector<Problem> &ps, const std::vector<int> &order, int pairs, bool tail) {
  std::vector<double> load(static_cast<size_t>(pairs), 0.0);
  int64_t total = 0;
  for (int i : order) total += int64_t(ps[size_t(i)].tiles_m) * ps[size_t(i)].tiles_n * ps[size_t(i)].splits;
  const int64_t T = total % pairs;
  const int64_t whole = tail ? total - T : total;
  int64_t u = 0;
  for (int i : order) {
    const Problem &p = ps[size_t(i)];
    const int64_t n = int64_t(p.tiles_m) * p.tiles_n * p.splits;
    for (int64_t j = 0; j < n; ++j, ++u) {
      const int split = int(j % p.splits);
      const double len = double((split + 1) * p.k_blocks / p.splits - split * p.k_blocks / p.splits);
      if (u < whole) {
        load[size_t(u % pairs)] += len;
      } else {  // two half-width units of this tile, on the next two pairs of the tail wave
        const int64_t h = whole + 2 * (u - whole);
        load[size_t(h % pairs)] += kHalfUnitCost * len;
        load[size_t((h + 1) % pairs)] += kHalfUnitCost * len;
      }
    }
  }
  return *std::max_element(load.begin(), load.end());
}

// Split counts and order of a group: every combination of split counts (1..8, at least 4
// k-blocks a unit) of its splittable products is modeled, products ordered by unit length,
// longest first; the score is the modeled time plus 3 % per extra split (each one more
// fp32 reduce-add of the product's output, and fewer operand reuses in L2; measured on the
// layer shapes, where the model alone over-splits).  Cached per group shape.
struct GroupPlan {
  std::vector<int> splits, order;
  bool tail = false;
};

GroupPlan plan_group(const std::vector<Problem> &base, const std::vector<bool> &may_split, int pairs) {
  static std::mutex mu;
  static std::map<std::vector<int64_t>, GroupPlan> cache;
  std::vector<int64_t> key{pairs};
  for (size_t i = 0; i < base.size(); ++i)
    key.insert(key.end(), {base[i].m_dim, base[i].n_dim, base[i].k_dim, int64_t(may_split[i])});
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  const int n = int(base.size());
  std::vector<std::vector<int>> opts(static_cast<size_t>(n));
  for (int i = 0; i < n; ++i) {
    opts[size_t(i)].push_back(1);
    if (may_split[size_t(i)])
      for (int s = 2; s <= 8 && base[size_t(i)].k_blocks / s >= 4; ++s) opts[size_t(i)].push_back(s);
  }
  const char *force = std::getenv("GTP_GROUP_SPLITS");  // a fixed split count (measurement sweeps)
  GroupPlan best;
  double best_score = 1e300;
  std::vector<size_t> idx(static_cast<size_t>(n), 0);
  while (true) {
    std::vector<Problem> ps = base;
    int extra = 0;
    bool skip = false;
    for (int i = 0; i < n; ++i) {
      int s = opts[size_t(i)][idx[size_t(i)]];
      if (force && may_split[size_t(i)]) {
        const int f = std::atoi(force);
        if (s != std::max(1, std::min(f, opts[size_t(i)].back()))) skip = true;
      }
      ps[size_t(i)].splits = s;
      extra += s - 1;
    }
    if (!skip) {
      std::vector<int> order(static_cast<size_t>(n));
      for (int i = 0; i < n; ++i) order[size_t(i)] = i;
      std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
        return ps[size_t(a)].k_blocks * ps[size_t(b)].splits > ps[size_t(b)].k_blocks * ps[size_t(a)].splits;
      });
      for (int t = 0; t < 2; ++t) {
        const Problem &last = ps[size_t(order.back())];
        int64_t total = 0;
        for (const Problem &p : ps) total += int64_t(p.tiles_m) * p.tiles_n * p.splits;
        const int64_t T = total % pairs;
        const bool can_tail = last.splits == 1 && T > 0 && 2 * T <= pairs &&
                              T <= int64_t(last.tiles_m) * last.tiles_n;
        if (t == 1 && !can_tail) break;
        const double score = group_makespan(ps, order, pairs, t == 1) * (1.0 + 0.03 * extra);
        if (score < best_score - 1e-9) {
          best_score = score;
          best.splits.assign(size_t(n), 1);
          for (int i = 0; i < n; ++i) best.splits[size_t(i)] = ps[size_t(i)].splits;
          best.order = order;
          best.tail = t == 1;
        }
      }
    }
    int i = 0;
    while (i < n && ++idx[size_t(i)] == opts[size_t(i)].size()) idx[size_t(i++)] = 0;
    if (i == n) break;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() >= 4096) cache.clear();  // a process that meets many group shapes plans them again
  cache.emplace(key, best);
  return best;
}

// Launches the products of `spec` (1 to grp::kMaxItems, each with more than 128 output rows)
// as one grouped CTA-pair kernel.  deterministic: no split contractions.
gtp_status run_group(const GroupSpec *spec, int n, bool deterministic, const gtp::DeviceInfo &dev,
                     cudaStream_t stream) {
  if (n < 1 || n > grp::kMaxItems) return gtp::fail(GTP_E_ARG, "a group holds 1 to %d products", grp::kMaxItems);
  static std::atomic<uint64_t> configured{0};
  if (gtp_status e = configure(gemm_bf16_group_kernel, pair::SMEM_TOTAL, configured, dev.device)) return e;
  const int pairs = max_pairs(gemm_bf16_pair_kernel<false, false, kStoreBf16, false>, dev);
  std::vector<Problem> base(static_cast<size_t>(n));
  std::vector<bool> may_split(static_cast<size_t>(n));
  for (int i = 0; i < n; ++i) {
    base[size_t(i)] = tile_problem(spec[i].o, true);
    base[size_t(i)].group_m = 1;
    base[size_t(i)].splits = 1;
    may_split[size_t(i)] = spec[i].may_split && !deterministic;
  }
  const GroupPlan plan = plan_group(base, may_split, pairs);
  grp::Args args;
  std::memset(&args, 0, sizeof(args));
  args.n = n;
  int32_t unit = 0;
  for (int j = 0; j < n; ++j) {
    const int i = plan.order[size_t(j)];
    const GroupSpec &sp = spec[i];
    grp::Maps &m = args.maps[j];
    if (gtp_status s = encode_maps(sp.o, sp.a_mn, sp.b_mn, sp.epi, true, m.a, m.b, m.bh, m.d)) return s;
    Problem p = base[size_t(i)];
    p.splits = plan.splits[size_t(i)];
    const int tiles = p.tiles_m * p.tiles_n;
    p.num_units = tiles * p.splits;
    finalize_problem(p);
    set_l2_hints(sp.o, p);
    p.direct = sp.o.d;
    if (j == n - 1 && plan.tail) {
      const int T = (unit + p.num_units) % pairs;
      p.tail_first = p.num_units - T;
      p.tail_half = 1;
      p.num_units = p.tail_first + 2 * T;
    }
    grp::Item &it = args.it[j];
    it.p = p;
    it.a_mn = sp.a_mn;
    it.b_mn = sp.b_mn;
    it.epi = sp.epi;
    it.unit_begin = unit;
    unit += p.num_units;
  }
  args.num_units = unit;
  const int grid = 2 * std::min(args.num_units, pairs);
  return gtp::launch_overlapped(gemm_bf16_group_kernel, grid, pair::kThreads, pair::SMEM_TOTAL, stream,
                                "gemm_bf16_group_kernel", args);
}

}  // namespace

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

namespace {

// Both wgrad entry points: with `split` the contraction may be split across CTA pairs
// (partial tiles meet through fp32 reduce-adds, in whatever order they land); without it
// every output tile is one CTA pair's fixed-order sum, reduce-added once per call.
gtp_status wgrad_entry(const void *dY, const void *X, float *grad_data, int64_t grad_offset, int64_t grad_numel_total,
                       int64_t M, int64_t N, int64_t K, gtp_dtype dt, gtp_stream stream, bool split) {
  gtp::clear_error();
  if (dt != GTP_BF16) return gtp::fail(GTP_E_DTYPE, "only GTP_BF16 is supported");
  if (gtp_status s = check_dims(M, N, K)) return s;
  if (grad_offset < 0 || grad_numel_total < 0) return gtp::fail(GTP_E_ARG, "negative offset or size");
  if (N * K > grad_numel_total - grad_offset)
    return gtp::fail(GTP_E_RANGE, "view [%lld, +%lld) exceeds the grad buffer (%lld)", (long long)grad_offset,
                     (long long)(N * K), (long long)grad_numel_total);
  if (M == 0 || N == 0 || K == 0) return GTP_OK;
  if (!dY || !X || !grad_data) return gtp::fail(GTP_E_ARG, "null pointer");
  if (!gtp::aligned16(dY) || !gtp::aligned16(X)) return gtp::fail(GTP_E_ALIGN, "dY and X must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(grad_data) & 3u) return gtp::fail(GTP_E_ALIGN, "grad_data must be 4-byte aligned");
  gtp::DeviceInfo dev;
  if (gtp_status s = gtp::require_sm103(&dev)) return s;
  // D = main_grad view [N, K], contraction M; A = dY [M, N] (MN-major), B = X [M, K] (MN-major).
  // A view that starts on a 16-byte boundary takes the TMA reduce-add; any other (the
  // unpadded default layout puts a parameter at any element) the register atomic adds.
  const Operands o{dY, X, grad_data + grad_offset, int(N), int(K), int(M)};
  if (gtp::aligned16(grad_data + grad_offset))
    return run_gemm<true, true, kReduceAddF32>(o, split, dev, gtp::as_stream(stream));
  return run_gemm<true, true, kReduceAddF32Direct>(o, split, dev, gtp::as_stream(stream));
}

}  // namespace

extern "C" gtp_status gtp_linear_wgrad_accum(const void *dY, const void *X, float *grad_data, int64_t grad_offset,
                                             int64_t grad_numel_total, int64_t M, int64_t N, int64_t K, gtp_dtype dt,
                                             gtp_stream stream) {
  return wgrad_entry(dY, X, grad_data, grad_offset, grad_numel_total, M, N, K, dt, stream, true);
}

extern "C" gtp_status gtp_linear_wgrad_accum_deterministic(const void *dY, const void *X, float *grad_data,
                                                           int64_t grad_offset, int64_t grad_numel_total, int64_t M,
                                                           int64_t N, int64_t K, gtp_dtype dt, gtp_stream stream) {
  return wgrad_entry(dY, X, grad_data, grad_offset, grad_numel_total, M, N, K, dt, stream, false);
}

extern "C" gtp_status gtp_linear_wgrad_accum_bf16(const void *dY, const void *X, void *grad_data, int64_t grad_offset,
                                                  int64_t grad_numel_total, int64_t M, int64_t N, int64_t K,
                                                  gtp_dtype dt, gtp_stream stream) {
  gtp::clear_error();
  if (dt != GTP_BF16) return gtp::fail(GTP_E_DTYPE, "only GTP_BF16 is supported");
  if (gtp_status s = check_dims(M, N, K)) return s;
  if (grad_offset < 0 || grad_numel_total < 0) return gtp::fail(GTP_E_ARG, "negative offset or size");
  if (N * K > grad_numel_total - grad_offset)
    return gtp::fail(GTP_E_RANGE, "view [%lld, +%lld) exceeds the grad buffer (%lld)", (long long)grad_offset,
                     (long long)(N * K), (long long)grad_numel_total);
  if (M == 0 || N == 0 || K == 0) return GTP_OK;
  if (!dY || !X || !grad_data) return gtp::fail(GTP_E_ARG, "null pointer");
  if (!gtp::aligned16(dY) || !gtp::aligned16(X)) return gtp::fail(GTP_E_ALIGN, "dY and X must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(grad_data) & 1u) return gtp::fail(GTP_E_ALIGN, "grad_data must be 2-byte aligned");
  gtp::DeviceInfo dev;
  if (gtp_status s = gtp::require_sm103(&dev)) return s;
  // D = the bf16 main_grad view [N, K]; one CTA owns each element (no split), which reads
  // it, adds its fp32 accumulator and writes the bf16 rounding of the sum
  return run_gemm<true, true, kAccumBf16>(
      {dY, X, static_cast<__nv_bfloat16 *>(grad_data) + grad_offset, int(N), int(K), int(M)}, false, dev,
      gtp::as_stream(stream));
}

namespace {

// What a grouped call does with one product, decided before anything is launched.
enum { kNothing = 0, kZeroFill = 1, kGroup = 2, kAlone = 3 };

struct Prepared {
  int action = kNothing;
  GroupSpec spec{};
  void *zero_ptr = nullptr;  // kZeroFill: the output, all of whose bytes become 0
  int64_t zero_bytes = 0;
};

// Validates one product as its single entry point does and classifies it: nothing to do
// (an empty output or contraction for wgrad), zeros (an empty contraction for fprop /
// dgrad), a unit of the grouped kernel, or a launch of its own (at most 128 output rows:
// the single-CTA kernel; or every product alone when GTP_GEMM_VARIANT picks a kernel).
gtp_status prepare_desc(const gtp_gemm_desc &d, Prepared &out) {
  if (d.reserved != 0) return gtp::fail(GTP_E_ARG, "reserved must be 0");
  if (d.dtype != GTP_BF16) return gtp::fail(GTP_E_DTYPE, "only GTP_BF16 is supported");
  if (gtp_status s = check_dims(d.M, d.N, d.K)) return s;
  const int64_t M = d.M, N = d.N, K = d.K;
  switch (d.kind) {
    case GTP_GEMM_FPROP:
      if (M == 0 || N == 0) return GTP_OK;
      if (!d.out || (K > 0 && (!d.a || !d.b))) return gtp::fail(GTP_E_ARG, "null pointer");
      if (!gtp::aligned16(d.out) || (K > 0 && (!gtp::aligned16(d.a) || !gtp::aligned16(d.b))))
        return gtp::fail(GTP_E_ALIGN, "pointers must be 16-byte aligned");
      if (K == 0) {
        out.action = kZeroFill;
        out.zero_ptr = d.out;
        out.zero_bytes = M * N * 2;
        return GTP_OK;
      }
      out.spec = {{d.a, d.b, d.out, int(M), int(N), int(K)}, false, false, kStoreBf16, false};
      break;
    case GTP_GEMM_DGRAD:
      if (M == 0 || K == 0) return GTP_OK;
      if (!d.out || (N > 0 && (!d.a || !d.b))) return gtp::fail(GTP_E_ARG, "null pointer");
      if (!gtp::aligned16(d.out) || (N > 0 && (!gtp::aligned16(d.a) || !gtp::aligned16(d.b))))
        return gtp::fail(GTP_E_ALIGN, "pointers must be 16-byte aligned");
      if (N == 0) {
        out.action = kZeroFill;
        out.zero_ptr = d.out;
        out.zero_bytes = M * K * 2;
        return GTP_OK;
      }
      out.spec = {{d.a, d.b, d.out, int(M), int(K), int(N)}, false, true, kStoreBf16, false};
      break;
    case GTP_GEMM_WGRAD_ACCUM: {
      if (d.grad_dtype != GTP_F32 && d.grad_dtype != GTP_BF16)
        return gtp::fail(GTP_E_DTYPE, "grad_dtype must be GTP_F32 or GTP_BF16");
      if (d.grad_offset < 0 || d.grad_numel_total < 0) return gtp::fail(GTP_E_ARG, "negative offset or size");
      if (N * K > d.grad_numel_total - d.grad_offset)
        return gtp::fail(GTP_E_RANGE, "view [%lld, +%lld) exceeds the grad buffer (%lld)", (long long)d.grad_offset,
                         (long long)(N * K), (long long)d.grad_numel_total);
      if (M == 0 || N == 0 || K == 0) return GTP_OK;
      if (!d.a || !d.b || !d.out) return gtp::fail(GTP_E_ARG, "null pointer");
      if (!gtp::aligned16(d.a) || !gtp::aligned16(d.b)) return gtp::fail(GTP_E_ALIGN, "dY and X must be 16-byte aligned");
      const bool bf16 = d.grad_dtype == GTP_BF16;
      if (reinterpret_cast<uintptr_t>(d.out) & (bf16 ? 1u : 3u))
        return gtp::fail(GTP_E_ALIGN, "grad_data must be aligned to its element");
      void *view = bf16 ? static_cast<void *>(static_cast<__nv_bfloat16 *>(d.out) + d.grad_offset)
                        : static_cast<void *>(static_cast<float *>(d.out) + d.grad_offset);
      // a bf16 buffer: the bf16 accumulate (never split); fp32: the TMA reduce-add where
      // TMA can address the view, else fp32 atomic adds
      const int epi = bf16 ? kAccumBf16 : gtp::aligned16(view) ? kReduceAddF32 : kReduceAddF32Direct;
      out.spec = {{d.a, d.b, view, int(N), int(K), int(M)}, true, true, epi, !bf16};
      break;
    }
    default:
      return gtp::fail(GTP_E_ARG, "unknown product kind %d", int(d.kind));
  }
  out.action = use_pair(out.spec.o.m_dim) && !std::getenv("GTP_GEMM_VARIANT") ? kGroup : kAlone;
  return GTP_OK;
}

gtp_status run_alone(const GroupSpec &g, bool deterministic, const gtp::DeviceInfo &dev, cudaStream_t st) {
  if (g.epi == kReduceAddF32) return run_gemm<true, true, kReduceAddF32>(g.o, !deterministic, dev, st);
  if (g.epi == kReduceAddF32Direct) return run_gemm<true, true, kReduceAddF32Direct>(g.o, !deterministic, dev, st);
  if (g.epi == kAccumBf16) return run_gemm<true, true, kAccumBf16>(g.o, false, dev, st);
  if (g.b_mn) return run_gemm<false, true, kStoreBf16>(g.o, false, dev, st);
  return run_gemm<false, false, kStoreBf16>(g.o, false, dev, st);
}

// The products of a group must be independent: an output that overlaps an input or
// another output is an argument error, found before anything is launched.  Inputs may be
// shared (a linear's dgrad and wgrad both read dY), and two fp32 WGRAD_ACCUM views may
// overlap (their fp32 additions commute).
gtp_status check_independent(const gtp_gemm_desc *descs, const Prepared *prep, int n) {
  struct Range {
    uintptr_t lo, hi;
    int product;
    const char *what;  // nullptr: an input
    bool f32_accum;
  };
  Range r[3 * grp::kMaxItems];
  int nr = 0;
  auto add = [&](const void *ptr, int64_t bytes, int i, const char *what, bool f32_accum) {
    if (!ptr || bytes <= 0) return;
    const uintptr_t lo = reinterpret_cast<uintptr_t>(ptr);
    r[nr++] = Range{lo, lo + uintptr_t(bytes), i, what, f32_accum};
  };
  for (int i = 0; i < n; ++i) {
    if (prep[i].action == kNothing) continue;
    const gtp_gemm_desc &d = descs[i];
    const int64_t M = d.M, N = d.N, K = d.K;
    if (d.kind == GTP_GEMM_FPROP) {
      add(d.a, M * K * 2, i, nullptr, false);
      add(d.b, N * K * 2, i, nullptr, false);
      add(d.out, M * N * 2, i, "output", false);
    } else if (d.kind == GTP_GEMM_DGRAD) {
      add(d.a, M * N * 2, i, nullptr, false);
      add(d.b, N * K * 2, i, nullptr, false);
      add(d.out, M * K * 2, i, "output", false);
    } else {
      const int64_t es = d.grad_dtype == GTP_BF16 ? 2 : 4;
      add(d.a, M * N * 2, i, nullptr, false);
      add(d.b, M * K * 2, i, nullptr, false);
      add(static_cast<const uint8_t *>(d.out) + d.grad_offset * es, N * K * es, i, "main_grad view",
          d.grad_dtype == GTP_F32);
    }
  }
  for (int i = 0; i < nr; ++i)
    for (int j = i + 1; j < nr; ++j) {
      if (!r[i].what && !r[j].what) continue;
      if (r[i].f32_accum && r[j].f32_accum) continue;
      if (r[i].lo < r[j].hi && r[j].lo < r[i].hi)
        return gtp::fail(GTP_E_ARG, "product %d's %s overlaps product %d's %s", r[i].product,
                         r[i].what ? r[i].what : "input", r[j].product, r[j].what ? r[j].what : "input");
    }
  return GTP_OK;
}

gtp_status grouped_entry(const gtp_gemm_desc *descs, int32_t n, int32_t flags, gtp_stream stream) {
  if (n < 0 || n > grp::kMaxItems) return gtp::fail(GTP_E_ARG, "n must lie in [0, %d]", grp::kMaxItems);
  if (n > 0 && !descs) return gtp::fail(GTP_E_ARG, "null descriptor array");
  if (flags & ~int32_t(GTP_GEMM_DETERMINISTIC)) return gtp::fail(GTP_E_ARG, "unknown flags 0x%x", unsigned(flags));
  Prepared prep[grp::kMaxItems];
  for (int i = 0; i < n; ++i)  // every argument is checked before anything is launched
    if (gtp_status s = prepare_desc(descs[i], prep[i])) return s;
  bool any = false;
  for (int i = 0; i < n; ++i) any = any || prep[i].action != kNothing;
  if (!any) return GTP_OK;
  if (gtp_status s = check_independent(descs, prep, n)) return s;
  const bool det = (flags & GTP_GEMM_DETERMINISTIC) != 0;
  gtp::DeviceInfo dev;
  if (gtp_status s = gtp::require_sm103(&dev)) return s;
  cudaStream_t st = gtp::as_stream(stream);
  GroupSpec group[grp::kMaxItems];
  int ng = 0;
  for (int i = 0; i < n; ++i) {
    gtp_status s = GTP_OK;
    if (prep[i].action == kZeroFill)
      s = gtp::launch_zero_bytes(prep[i].zero_ptr, prep[i].zero_bytes, st, dev.sm_count);
    else if (prep[i].action == kAlone)
      s = run_alone(prep[i].spec, det, dev, st);
    else if (prep[i].action == kGroup)
      group[ng++] = prep[i].spec;
    if (s) return s;
  }
  return ng ? run_group(group, ng, det, dev, st) : GTP_OK;
}

}  // namespace

extern "C" gtp_status gtp_linear_grouped(const gtp_gemm_desc *descs, int32_t n, int32_t flags, gtp_stream stream) {
  gtp::clear_error();
  return grouped_entry(descs, n, flags, stream);
}

extern "C" gtp_status gtp_linear_backward(const void *dY, const void *X, const void *W, void *dX, float *grad_data,
                                          int64_t grad_offset, int64_t grad_numel_total, int64_t M, int64_t N,
                                          int64_t K, gtp_dtype dt, int32_t flags, gtp_stream stream) {
  gtp::clear_error();
  gtp_gemm_desc d[2] = {};
  d[0].kind = GTP_GEMM_DGRAD;
  d[0].a = dY;
  d[0].b = W;
  d[0].out = dX;
  d[1].kind = GTP_GEMM_WGRAD_ACCUM;
  d[1].grad_dtype = GTP_F32;
  d[1].a = dY;
  d[1].b = X;
  d[1].out = grad_data;
  d[1].grad_offset = grad_offset;
  d[1].grad_numel_total = grad_numel_total;
  for (gtp_gemm_desc &x : d) {
    x.dtype = dt;
    x.M = M;
    x.N = N;
    x.K = K;
  }
  return grouped_entry(d, 2, flags, stream);
}

namespace {

// Failure-detection self-test: one thread waits, with the library's bounded wait and a
// short limit, on an mbarrier that nothing ever arrives on.  The wait runs out, raises the
// CTA's abort flag and bit 0x100 of this unit's wait-timeout word, and the kernel returns
// normally: the context stays usable and the host reads the bit with gtp_wait_timeouts.
__global__ void wait_timeout_selftest_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_limit(&bar, 0, &abort_flag, &g_gtp_wait_timeouts, 0x100u, limit_ns);
}

}  // namespace

extern "C" gtp_status gtp_selftest_wait_timeout(int64_t limit_ns, gtp_stream stream) {
  gtp::clear_error();
  if (limit_ns < 1000 || limit_ns > 100000000)
    return gtp::fail(GTP_E_ARG, "limit_ns must lie in [1e3, 1e8] (1 us .. 100 ms)");
  gtp::DeviceInfo dev;
  if (gtp_status s = gtp::require_sm103(&dev)) return s;
  wait_timeout_selftest_kernel<<<1, 32, 0, gtp::as_stream(stream)>>>(uint64_t(limit_ns));
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return gtp::fail(GTP_E_CUDA, "wait self-test launch: %s", cudaGetErrorString(e));
  return GTP_OK;
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
  unsigned int w = 0;  // the block-scaled kernels keep their own word
  if (gtp_status s = gtp::blockscaled_wait_word(&w, reset != 0)) return s;
  *flags = v | w;
  return GTP_OK;
}

