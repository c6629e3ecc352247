// The block-scaled GEMMs on the 5th-generation tensor cores: MXFP8 (forward, dgrad and
// wgrad-accumulate on the rowwise / columnwise views) and NVFP4 (forward).
//
// Page: "Generalized Tensor Parallelism (GTP)" (Megatron-Core developer guide), §1.3
// (native MXFP8 / NVFP4 weights, blocks of 32 / 16 elements with one scale each) on top of
// the linear layer's three products ("01 · ColumnParallelLinear / RowParallelLinear and the
// core autograd" (llm-infra-atlas), §4.1, §4.2).
#include "gemm_common.cuh"
#include "nv_block.cuh"

namespace {

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

// A TMA tile store with an L2 cache policy (createpolicy), for an output streamed once that
// should not push the operands every wave re-reads out of L2.
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap *map, const void *src, int32_t c0, int32_t c1,
                                                  uint64_t policy) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], %4;" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(gtp::ptx::smem_u32(src)), "r"(c0), "r"(c1), "l"(policy)
               : "memory");
}

// The block-scaled kernel keeps one accumulator (the scale columns take the rest of tensor
// memory), so its epilogue runs 8 warps, two per 32-lane quarter, each holding half of its
// rows' 256 columns in registers: the accumulator is released as soon as it has been read,
// and the conversion and stores of one tile overlap the main loop of the next.
constexpr int kBsEpiWarps = 8;
constexpr int kBsThreads = 64 + 32 * kBsEpiWarps;

constexpr int kBsEpiBuf = 32 * 64;  // per epilogue warp: 32 rows x 64 bytes (64-byte swizzle)

// S: operand stages of the one-CTA kernel (the CTA-pair kernel's traits follow further
// down).  The ring is what keeps loads in flight, so the staging buffers stay small to
// leave room for it; but shared memory also sets the L1 size left over, and a long
// contraction re-reads each row's scale words from L1 stage after stage (this kernel
// gathers them with loads).  MXFP8 runs 4 stages on short contractions and 3 on long ones
// (the host picks); NVFP4, whose scale words take 6 KB per stage, always runs 3.
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
  } else if (warp == 1) {  // ------------- MMA issuer: the whole warp waits, one elected lane issues
    int stage = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
      int tm, tn, kb0, kb1;
      decode_unit(p, u, tm, tn, kb0, kb1);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(tempty, acc_phase ^ 1u, abort_flag, err, 0x2u))) break;
      tc_fence_after();
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[stage], phase, abort_flag, err, 0x4u))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (elect_one_sync()) {
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
        }
        __syncwarp();
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (elect_one_sync()) mma_commit(tfull);
      __syncwarp();
      acc_phase ^= 1u;
    }
    if (elect_one_sync()) mma_commit(drain);
    __syncwarp();
    if (lane == 0) drain_wait(drain, 0);
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
      // the next tile's MMAs may overwrite the accumulator: the loads above have completed
      // (wait::ld); a release would also wait for this warp's earlier stores in flight
      if (lane == 0) mbar_arrive_relaxed(tempty);
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

// ----------------------------------------------------------- block-scaled, CTA pair
//
// The same products on 256x256 tiles computed by a CTA pair with M = 256 block-scaled
// MMAs (cta_group::2): each CTA stages its 128 rows of A and its 128 rows of B (half the
// tile's B), so an SM moves 32 KB of operands per stage instead of 48 and keeps more
// stages in flight.  The even CTA issues the MMAs and the scale copies into both CTAs'
// tensor memory (tcgen05.cp.cta_group::2: each CTA's copy comes from its own shared
// memory): each CTA holds the scale words of its own A rows and of all 256 B rows.  The
// even CTA's full barrier counts both CTAs' operand bytes (the TMA loads complete on it)
// and one arrival from each CTA's scale warps, made after that CTA's scale words of the
// stage are in shared memory.
// TSF: the scale rows arrive by tensor copies (16-byte aligned rows and base); otherwise one
// scale warp gathers the words with loads into a register ring (as the one-CTA kernel
// does), which a weight's scale view inside a native MXFP8 buffer needs (its rows start on
// the 64-element parameter alignment: 2-byte aligned scale bytes).
template <int FMT, int S, bool TSF = true, bool TILED = false>
struct BlockScaledPair {
  using F1 = BlockScaled<FMT, 3>;  // per-stage geometry shared with the one-CTA kernel
  static constexpr bool SF_TMA = TSF;
  // TILED: the scale arrays come in the tiled layout (gtp_sf_tile): a stage's words of 128
  // rows are one contiguous 512-byte atom per word, already in the order tcgen05.cp reads,
  // so the producer copies them with the operands (three boxes a stage) and no scale warp
  // runs.  The B atoms of a stage land as [row-tile half][word] (two boxes of WORDS atoms).
  static constexpr bool SF_TILED = TILED;
  static constexpr int PREFETCH = F1::PREFETCH;  // gather path: stages of scale words in registers
  static constexpr int STAGES = S;
  static constexpr int WORDS = F1::WORDS, K_STAGE = F1::K_STAGE, BK = F1::BK, UKB = F1::UKB;
  static constexpr int SF_BLOCK = F1::SF_BLOCK;
  static constexpr int BMP = 256, BMC = 128, BNC = 128;
  static constexpr int A_STAGE = BMC * BK;  // 16 KB
  static constexpr int B_STAGE = BNC * BK;  // 16 KB
  static constexpr int SFA_STAGE = BMC * 4 * WORDS;
  static constexpr int SFB_STAGE = BN * 4 * WORDS;  // all 256 B rows
  static constexpr int STAGE_TX = A_STAGE + B_STAGE;
  static constexpr int SMEM_OPS = STAGES * (A_STAGE + B_STAGE);
  // per stage, one slot: the A words, then the B words, in the layout tcgen05.cp reads
  static constexpr int SF_SLOT = SFA_STAGE + SFB_STAGE;
  static constexpr int SMEM_SF = (STAGES * SF_SLOT + 1023) / 1024 * 1024;
  // Scale bytes arrive by TMA, 16 per row (a 16-byte box is the narrowest a tensor copy
  // takes): GROUP stages' worth per landing slot (4 MXFP8 stages of one word, or one NVFP4
  // stage of four), this CTA's 128 A rows and the tile's 256 B rows.
  static constexpr int GROUP = 4 / WORDS;
  static constexpr int LAND_A = BMC * 16, LAND_B = BN * 16, LAND_BYTES = LAND_A + LAND_B;
  // NVFP4 moves 6 KB of scale words a stage: two scale warps take alternate groups (one
  // warp's serial chain of shared-memory steps measured longer than the stage's MMAs);
  // MXFP8's one word a stage needs one.  LAND slots per scale warp, as many as fit.
  // NVFP4's 16 bytes of a row are exactly one stage, and a stage's landed rows take as many
  // bytes as its words in the copy layout (SF_SLOT == LAND_BYTES): the producer lands them
  // straight in the stage's slot, next to the stage's operands, and a scale warp permutes
  // them in place (two warps, alternate stages).  MXFP8's 16 bytes of a row span four
  // stages: its scale warp lands them in a separate slot and hands out one word a stage.
  static constexpr bool SF_INPLACE = TSF && FMT == kNvfp4 && !TILED;
  // tiled scales: one warp issues the stage's three scale copies beside the operand producer
  static constexpr int SCALE_WARPS = SF_INPLACE ? 2 : 1;
  static constexpr int LAND = (TILED || !TSF || SF_INPLACE) ? 0 : S >= 6 ? 1 : 2;
  static constexpr int SMEM_LAND = SCALE_WARPS * LAND * LAND_BYTES;
  static constexpr int LFULL = SF_INPLACE ? STAGES : SCALE_WARPS * LAND;  // landing barriers
  static_assert(!SF_INPLACE || SF_SLOT == LAND_BYTES, "in-place slots");
  static constexpr int THREADS = kBsThreads + 32 * SCALE_WARPS;
  static constexpr int SMEM_EPI = kBsEpiWarps * kBsEpiBuf;
  static constexpr int SMEM_TOTAL = SMEM_OPS + SMEM_SF + SMEM_LAND + SMEM_EPI + SMEM_CTRL + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t SFA_COL = BN;
  static constexpr uint32_t SFB_COL = BN + 4 * WORDS * STAGES;
  static_assert(SMEM_TOTAL <= 232448, "shared memory per block");
  static_assert(SFB_COL + 8 * WORDS * STAGES <= TMEM_COLS, "tensor memory columns");
  static_assert((SMEM_OPS + SMEM_SF + SMEM_LAND) % 1024 == 0, "staging buffers 1024-byte aligned");
  static_assert((2 * STAGES + 3 + LFULL) * 8 + 8 <= SMEM_CTRL, "barriers");
};

template <int FMT, int EPI, int S, bool TSF, bool TILED>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(BlockScaledPair<FMT, S, TSF, TILED>::THREADS, 1)
    gemm_blockscaled_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                                 const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmSA,
                                 const __grid_constant__ CUtensorMap tmSB, const uint8_t *__restrict__ sfa_g,
                                 const uint8_t *__restrict__ sfb_g, const float *__restrict__ a_amax,
                                 const float *__restrict__ b_amax, const Problem p) {
  using F = BlockScaledPair<FMT, S, TSF, TILED>;
  constexpr int STAGES = F::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sA = smem;
  uint8_t *sB = sA + STAGES * F::A_STAGE;
  uint8_t *sSF = smem + F::SMEM_OPS;  // per stage: SFA words, then SFB words
  auto sfa_of = [&](int s) { return reinterpret_cast<uint32_t *>(sSF + s * F::SF_SLOT); };
  auto sfb_of = [&](int s) { return reinterpret_cast<uint32_t *>(sSF + s * F::SF_SLOT + F::SFA_STAGE); };
  uint8_t *sLand = smem + F::SMEM_OPS + F::SMEM_SF;  // scale bytes as the tensor copies land them
  uint8_t *sEpi = sLand + F::SMEM_LAND;
  uint64_t *full = reinterpret_cast<uint64_t *>(sEpi + F::SMEM_EPI);
  uint64_t *empty = full + STAGES;
  uint64_t *tfull = empty + STAGES;
  uint64_t *tempty = tfull + 1;
  uint64_t *drain = tempty + 1;
  uint64_t *lfull = drain + 1;  // a landing slot's scale bytes have arrived
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(lfull + F::LFULL);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // the even CTA's expect_tx arrival (both CTAs' operand bytes) and one arrival from
      // each CTA's scale warps once that CTA's scale words of the stage are in place (tiled
      // scales: the expect_tx arrival alone, the scale bytes counted with the operands)
      mbar_init(&full[s], F::SF_TILED ? 1 : 3);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < F::LFULL; ++s) mbar_init(&lfull[s], 1);
    mbar_init(tfull, 1);
    mbar_init(tempty, 2 * kBsEpiWarps);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmD);
    if (TSF) {
      tma_prefetch_desc(&tmSA);
      tma_prefetch_desc(&tmSB);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, F::TMEM_COLS);
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
  // the pair works through units pair, pair + npairs, ... (the one-CTA iterator, per pair)
  const int pair_id = int(blockIdx.x >> 1), npairs = int(gridDim.x >> 1);

  // Roles: warp 0 (one lane) issues the operand copies, warp 1 the MMAs (even CTA), warps
  // 2 .. 2 + kBsEpiWarps - 1 the epilogue, the last one or two warps the scale words.  The
  // operand copies of a stage go as soon as the MMAs have freed it; each CTA's scale warp
  // arrives on the even CTA's full barrier once that CTA's words of the stage are in place.
  constexpr int kScaleWarp = 2 + kBsEpiWarps;
  if (warp == 0) {  // ------------------------------------------ operand producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int armed[STAGES], armed_l[STAGES];  // parities of copies in flight (full, landing)
      for (int s = 0; s < STAGES; ++s) armed[s] = armed_l[s] = -1;
      const uint32_t full0 = mapa_shared(&full[0], 0);
      for (int u = pair_id; u < p.num_units; u += npairs) {
        int tm, tn, kb0, kb1;
        decode_unit(p, u, tm, tn, kb0, kb1);
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          // the operands go as soon as the stage is free: the scale warps signal the full
          // barrier themselves (waiting for them here cost the copies 400-1000 cycles of
          // their lead a stage)
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, err, 0x1u)) {
            ok = false;
            break;
          }
          const uint32_t bar = full0 + uint32_t(stage) * 8u;
          if constexpr (F::SF_INPLACE) {  // this CTA's scale rows of the stage, into its slot
            uint8_t *slot = sSF + stage * F::SF_SLOT;
            mbar_arrive_expect_tx_relaxed(&lfull[stage], F::SF_SLOT);
            // this CTA's A rows are rows 128 * (2 tm + rank) ..; B rows are the whole tile's
            tma_load_2d(&tmSA, &lfull[stage], slot, 16 * kb, (2 * tm + int(rank)) * BM);
            tma_load_2d(&tmSB, &lfull[stage], slot + F::SFA_STAGE, 16 * kb, tn * BN);
            armed_l[stage] = int(phase);
          }
          if (rank == 0) {  // the even CTA's barrier counts both CTAs' bytes
            mbar_arrive_expect_tx(&full[stage], 2 * (F::STAGE_TX + (F::SF_TILED ? F::SF_SLOT : 0)));
            armed[stage] = int(phase);
          }
          tma_load_2d_pair(&tmA, bar, sA + stage * F::A_STAGE, kb * F::BK, tm * F::BMP + F::BMC * int(rank));
          tma_load_2d_pair(&tmB, bar, sB + stage * F::B_STAGE, kb * F::BK, tn * BN + F::BNC * int(rank));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      for (int s = 0; s < STAGES; ++s) {
        if (armed[s] >= 0) drain_wait(&full[s], uint32_t(armed[s]));
        if (armed_l[s] >= 0) drain_wait(&lfull[s], uint32_t(armed_l[s]));
      }
    }
  } else if (warp >= kScaleWarp) {  // --------------------------------- scale warps (both CTAs)
    if constexpr (F::SF_TILED) {
      // The scale atoms arrive in the copy layout, on the stage's full barrier, which the
      // even CTA's operand producer arms for them too: this warp only issues the three
      // copies a stage (this CTA's A rows, both B halves) beside the operand producer's two.
      // One thread issuing all five fell behind the MMAs.
      if (lane == 0) {
        const uint32_t full0 = mapa_shared(&full[0], 0);
        const int wrow = p.k_dim / (4 * F::SF_BLOCK);  // atoms per 128-row tile
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int u = pair_id; ok && u < p.num_units; u += npairs) {
          int tm, tn, kb0, kb1;
          decode_unit(p, u, tm, tn, kb0, kb1);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, err, 0x1u)) {
              ok = false;
              break;
            }
            const uint32_t bar = full0 + uint32_t(stage) * 8u;
            uint8_t *slot = sSF + stage * F::SF_SLOT;
            const int w0 = kb * F::WORDS;
            tma_load_2d_pair(&tmSA, bar, slot, 0, (2 * tm + int(rank)) * wrow + w0);
            tma_load_2d_pair(&tmSB, bar, slot + F::SFA_STAGE, 0, 2 * tn * wrow + w0);
            tma_load_2d_pair(&tmSB, bar, slot + F::SFA_STAGE + 512 * F::WORDS, 0, (2 * tn + 1) * wrow + w0);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
    } else if constexpr (!F::SF_TMA) {
    // Gather path: the words of the next PREFETCH stages sit in registers (loads issued
    // ahead); each stage's words go to the tcgen05.cp layout once the MMAs have freed it.
    const uint32_t full0 = mapa_shared(&full[0], 0);
    const int64_t sf_row_bytes = p.k_dim / F::SF_BLOCK;
    constexpr int D = F::PREFETCH;
    ScaleRegs<F::WORDS> ring[D];
    int stage = 0;
    uint32_t phase = 0;
    int lu = pair_id, ltm = 0, ltn = 0, lkb = 0, lkb1 = 0;  // the loader's position
    int su = pair_id, stm = 0, stn = 0, skb = 0, skb1 = 0;  // the publisher's position
    if (lu < p.num_units) decode_unit(p, lu, ltm, ltn, lkb, lkb1);
    if (su < p.num_units) decode_unit(p, su, stm, stn, skb, skb1);
    auto next = [&](int &u, int &tm, int &tn, int &kb, int &kb1) {
      if (++kb == kb1) {
        u += npairs;
        if (u < p.num_units) decode_unit(p, u, tm, tn, kb, kb1);
      }
    };
#pragma unroll
    for (int d = 0; d < D; ++d)
      if (lu < p.num_units) {
        // this CTA's A rows are rows 128 * (2 tm + rank) ..; B rows are the whole tile's
        load_scales(ring[d], sfa_g, sfb_g, sf_row_bytes, p, 2 * ltm + int(rank), ltn, lkb, lane);
        next(lu, ltm, ltn, lkb, lkb1);
      }
    bool ok = true;
    while (ok && su < p.num_units) {
#pragma unroll
      for (int d = 0; d < D; ++d) {
        if (su >= p.num_units) break;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&empty[stage], phase ^ 1u, abort_flag, err, 0x1u))) {
          ok = false;
          break;
        }
        store_scales(ring[d], sfa_of(stage), sfb_of(stage), lane);
        fence_proxy_async_smem();  // the scale words are read by tcgen05.cp (async proxy)
        __syncwarp();
        if (lane == 0) {  // as on the tensor-copy path below
          if (rank == 0)
            mbar_arrive(&full[stage]);
          else
            mbar_arrive_cluster_relaxed(full0 + uint32_t(stage) * 8u);
        }
        if (lu < p.num_units) {
          load_scales(ring[d], sfa_g, sfb_g, sf_row_bytes, p, 2 * ltm + int(rank), ltn, lkb, lane);
          next(lu, ltm, ltn, lkb, lkb1);
        }
        next(su, stm, stn, skb, skb1);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    } else if constexpr (F::SF_INPLACE) {
    // The producer has landed this CTA's scale rows of each stage in the stage's slot; the
    // warp that owns the stage (stages alternate between the two) reads its lanes' rows,
    // writes the same bytes back in the layout tcgen05.cp reads, and signals the stage.
    constexpr int SW = F::SCALE_WARPS;
    const int sw = warp - kScaleWarp;
    const uint32_t full0 = mapa_shared(&full[0], 0);
    int stage = 0, gi = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int u = pair_id; ok && u < p.num_units; u += npairs) {
      int tm, tn, kb0, kb1;
      decode_unit(p, u, tm, tn, kb0, kb1);
      for (int kb = kb0; kb < kb1; ++kb, ++gi) {
        if (gi % SW == sw) {
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(&lfull[stage], phase, abort_flag, err, 0x1u))) {
            ok = false;
            break;
          }
          const uint8_t *slot = sSF + stage * F::SF_SLOT;
          ScaleRegs<4> R;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 v = *reinterpret_cast<const uint4 *>(slot + 16 * (32 * c + lane));
            R.a[c][0] = v.x, R.a[c][1] = v.y, R.a[c][2] = v.z, R.a[c][3] = v.w;
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4 v =
                *reinterpret_cast<const uint4 *>(slot + F::SFA_STAGE + 16 * (128 * (i >> 2) + 32 * (i & 3) + lane));
            R.b[i][0] = v.x, R.b[i][1] = v.y, R.b[i][2] = v.z, R.b[i][3] = v.w;
          }
          __syncwarp();  // every lane has read the landed rows before any lane overwrites them
          store_scales(R, sfa_of(stage), sfb_of(stage), lane);
          fence_proxy_async_smem();  // the scale words are read by tcgen05.cp (async proxy)
          __syncwarp();
          if (lane == 0) {  // as on the other scale paths
            if (rank == 0)
              mbar_arrive(&full[stage]);
            else
              mbar_arrive_cluster_relaxed(full0 + uint32_t(stage) * 8u);
          }
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    } else {
    // The loader fetches groups of scale bytes into the landing ring by TMA; the publisher
    // takes each group's words into registers, then hands every stage's words to the
    // layout tcgen05.cp reads as soon as the MMAs have freed that stage.  Lane 31 issues
    // the copies and lane 0 the stage signals: a release arrive waits for the arriving
    // thread's bulk copies in flight (measured: ~800 cycles a stage when one lane did both).
    // With two scale warps, warp sw takes the groups g (counted over the pair's whole
    // sequence) with g % 2 == sw, each into its own landing slots.
    constexpr int G = F::GROUP, L = F::LAND, SW = F::SCALE_WARPS;
    const int sw = warp - kScaleWarp;
    const uint32_t full0 = mapa_shared(&full[0], 0);
    uint64_t *my_lfull = lfull + sw * L;
    uint8_t *my_land = sLand + sw * L * F::LAND_BYTES;
    int lu = pair_id, ltm = 0, ltn = 0, lg = 0, lg1 = 0, lgi = 0;  // the loader's next group
    auto lstart = [&]() {
      if (lu < p.num_units) {
        int kb0, kb1;
        decode_unit(p, lu, ltm, ltn, kb0, kb1);
        lg = kb0 / G;
        lg1 = (kb1 - 1) / G + 1;
      }
    };
    auto lnext = [&]() {
      do {
        ++lgi;
        if (++lg == lg1) {
          lu += npairs;
          lstart();
        }
      } while (SW > 1 && lu < p.num_units && lgi % SW != sw);
    };
    int armed[L];  // parity of a slot's load in flight, -1 when none
    auto fetch = [&](int slot, uint32_t parity) {
      if (lu >= p.num_units) return;
      if (lane == 31) {
        uint8_t *dst = my_land + slot * F::LAND_BYTES;
        mbar_arrive_expect_tx_relaxed(&my_lfull[slot], F::LAND_BYTES);
        // this CTA's A rows are rows 128 * (2 tm + rank) ..; B rows are the whole tile's
        tma_load_2d(&tmSA, &my_lfull[slot], dst, 16 * lg, (2 * ltm + int(rank)) * BM);
        tma_load_2d(&tmSB, &my_lfull[slot], dst + F::LAND_A, 16 * lg, ltn * BN);
      }
      armed[slot] = int(parity);
      lnext();
    };
    lstart();
    if (SW > 1 && sw != 0) {  // the loader starts at this warp's first group
      lgi = -1;
      lg -= 1;  // lnext() steps to group 0 first
      lnext();
    }
    for (int s = 0; s < L; ++s) {
      armed[s] = -1;
      fetch(s, 0u);
    }
    int stage = 0, gslot = 0, su = pair_id, stm = 0, stn = 0, skb = 0, skb1 = 0, pgi = 0;
    uint32_t phase = 0, gphase = 0;
    if (su < p.num_units) decode_unit(p, su, stm, stn, skb, skb1);
    bool ok = true;
    while (ok && su < p.num_units) {  // one group a pass: it starts at stage (su, skb)
      if (SW > 1 && (pgi++) % SW != sw) {  // another warp's group: step over its stages
        do {
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          if (++skb == skb1) {
            su += npairs;
            if (su < p.num_units) decode_unit(p, su, stm, stn, skb, skb1);
            break;
          }
        } while (skb % G != 0);
        continue;
      }
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&my_lfull[gslot], gphase, abort_flag, err, 0x1u))) break;
      armed[gslot] = -1;
      ScaleRegs<4> R;  // the group's 16 bytes of each of this lane's rows
      const uint8_t *la = my_land + gslot * F::LAND_BYTES;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint4 v = *reinterpret_cast<const uint4 *>(la + 16 * (32 * c + lane));
        R.a[c][0] = v.x, R.a[c][1] = v.y, R.a[c][2] = v.z, R.a[c][3] = v.w;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 v = *reinterpret_cast<const uint4 *>(la + F::LAND_A + 16 * (128 * (i >> 2) + 32 * (i & 3) + lane));
        R.b[i][0] = v.x, R.b[i][1] = v.y, R.b[i][2] = v.z, R.b[i][3] = v.w;
      }
      // the slot is refilled after the group's first stage is published: by then every
      // lane has stored words of each of its loads (so the reads are complete), and that
      // stage's proxy fence orders them before the refill
      const int fslot = gslot;
      const uint32_t fparity = gphase ^ 1u;
      bool refilled = false;
      if (++gslot == L) {
        gslot = 0;
        gphase ^= 1u;
      }
      // the group's stages, word j of each row for stage j (a unit may start or end inside
      // a group; word indices stay compile-time constants so the words stay in registers)
      bool more = true;
#pragma unroll
      for (int j = 0; j < G; ++j) {
        if (!more || skb % G != j) continue;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&empty[stage], phase ^ 1u, abort_flag, err, 0x1u))) {
          ok = more = false;
          continue;
        }
        if constexpr (F::WORDS == 4) {
          store_scales(R, sfa_of(stage), sfb_of(stage), lane);
        } else {
          ScaleRegs<1> W;
#pragma unroll
          for (int c = 0; c < 4; ++c) W.a[c][0] = R.a[c][j];
#pragma unroll
          for (int i = 0; i < 8; ++i) W.b[i][0] = R.b[i][j];
          store_scales(W, sfa_of(stage), sfb_of(stage), lane);
        }
        fence_proxy_async_smem();  // the scale words are read by tcgen05.cp (async proxy)
        __syncwarp();
        // the even CTA's full barrier: a local release, or from the odd CTA a relaxed
        // cluster-scope arrive (a cluster-scope release measured 2.5x slower on the whole
        // kernel).  Every lane's proxy fence has made its words visible to the async proxy
        // and the warp barrier orders that before lane 0's arrive; the only reader is the
        // odd CTA's own tensor-memory copy, which the even CTA issues after the barrier.
        if (lane == 0) {
          if (rank == 0)
            mbar_arrive(&full[stage]);
          else
            mbar_arrive_cluster_relaxed(full0 + uint32_t(stage) * 8u);
        }
        if (!refilled) {
          fetch(fslot, fparity);
          refilled = true;
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
        if (++skb == skb1) {  // the unit ends: the next group is the next unit's
          su += npairs;
          if (su < p.num_units) decode_unit(p, su, stm, stn, skb, skb1);
          more = false;
        } else if (skb % G == 0) {
          more = false;
        }
      }
    }
    if (lane == 0)  // no tensor copy may still be writing this CTA's memory when it exits
      for (int s = 0; s < L; ++s)
        if (armed[s] >= 0) drain_wait(&my_lfull[s], uint32_t(armed[s]));
    }
  } else if (warp == 1) {  // -------- MMA issuer (even CTA only): the whole warp waits, one elected lane issues
    if (rank == 0) {
      auto copy_scales = [&](int s) {
        const uint32_t sfa_t = tmem_base + F::SFA_COL + 4 * F::WORDS * s;
        const uint32_t sfb_t = tmem_base + F::SFB_COL + 8 * F::WORDS * s;
        const uint32_t *fa = sfa_of(s);
        const uint32_t *fb = sfb_of(s);
#pragma unroll
        for (int w = 0; w < F::WORDS; ++w) {
          tmem_cp_32x128b_warpx4_pair(sfa_t + 4 * w, sdesc_noswizzle_rows16(smem_u32(fa + 128 * w)));
          // B rows 0-127 and 128-255 of word w: atoms [w][half], or [half][w] when tiled
          const int b0 = F::SF_TILED ? w : 2 * w, b1 = F::SF_TILED ? F::WORDS + w : 2 * w + 1;
          tmem_cp_32x128b_warpx4_pair(sfb_t + 8 * w, sdesc_noswizzle_rows16(smem_u32(fb + 128 * b0)));
          tmem_cp_32x128b_warpx4_pair(sfb_t + 8 * w + 4, sdesc_noswizzle_rows16(smem_u32(fb + 128 * b1)));
        }
      };
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int u = pair_id; ok && u < p.num_units; u += npairs) {
        int tm, tn, kb0, kb1;
        decode_unit(p, u, tm, tn, kb0, kb1);
        // the tile's first scale copies need only their stage, not the accumulator: issued
        // before the epilogue releases it, they run while the previous tile drains
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[stage], phase, abort_flag, err, 0x4u))) break;
        tc_fence_after();
        if (elect_one_sync()) copy_scales(stage);
        __syncwarp();
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(tempty, acc_phase ^ 1u, abort_flag, err, 0x2u))) break;
        tc_fence_after();
        for (int kb = kb0; kb < kb1; ++kb) {
          if (kb > kb0) {
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[stage], phase, abort_flag, err, 0x4u))) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          if (elect_one_sync()) {
            // each later stage's scale copy goes right before its own MMAs: issuing it a
            // stage early (when that stage had already landed) measured slower
            if (kb > kb0) copy_scales(stage);
            const uint32_t sfa_t = tmem_base + F::SFA_COL + 4 * F::WORDS * stage;
            const uint32_t sfb_t = tmem_base + F::SFB_COL + 8 * F::WORDS * stage;
            const uint32_t a0 = smem_u32(sA + stage * F::A_STAGE);
            const uint32_t b0 = smem_u32(sB + stage * F::B_STAGE);
#pragma unroll
            for (int k = 0; k < F::BK / F::UKB; ++k) {
              const uint64_t ad = sdesc_sw128(a0 + k * F::UKB, 16, 1024);
              const uint64_t bd = sdesc_sw128(b0 + k * F::UKB, 16, 1024);
              const uint32_t acc = (kb > kb0 || k > 0) ? 1u : 0u;
              if (FMT == kMxfp8)
                mma_mxf8_block_scale_pair(tmem_base, ad, bd, idesc_mxf8_e4m3(F::BMP, BN, uint32_t(k)), sfa_t, sfb_t,
                                          acc);
              else
                mma_nvf4_block_scale_pair(tmem_base, ad, bd, idesc_nvf4_e2m1(F::BMP, BN), sfa_t + 4 * k,
                                          sfb_t + 8 * k, acc);
            }
            mma_commit_pair(&empty[stage], 0x3);  // frees the stage in both CTAs
          }
          __syncwarp();
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (elect_one_sync()) mma_commit_pair(tfull, 0x3);  // both CTAs' epilogues may read their rows
        __syncwarp();
        acc_phase ^= 1u;
      }
      if (elect_one_sync()) mma_commit_pair(drain, 0x3);  // both CTAs learn when every MMA has finished
      __syncwarp();
    }
    if (lane == 0) drain_wait(drain, 0);
  } else if (warp < kScaleWarp) {  // ---------------------------------------- epilogue (both CTAs)
    const int ew = warp - 2;
    const int quarter = warp & 3;
    const int half = ew >> 2;
    uint8_t *buf = sEpi + ew * kBsEpiBuf;
    uint32_t acc_phase = 0;
    const uint32_t tempty0 = mapa_shared(tempty, 0);
    // bf16 outputs go out with an L2 evict_first policy: the fc1 forward writes 134 MB, more
    // than L2, while both operands (16-34 MB) are re-read by every wave; NVFP4 fc1 forward
    // 54.0 -> 51.9 us, MXFP8 82 -> 81 us
    const uint64_t pol_out = l2_policy(1);
    float alpha = 1.f;
    if (FMT == kNvfp4)
      alpha = float(1.0 / (double(gtp::nv::tensor_scale(__ldg(a_amax))) * double(gtp::nv::tensor_scale(__ldg(b_amax)))));
    for (int u = pair_id; u < p.num_units; u += npairs) {
      int tm, tn, kb0, kb1;
      decode_unit(p, u, tm, tn, kb0, kb1);
      const bool ok = mbar_wait(tfull, acc_phase, abort_flag, err, 0x8u);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
      tc_fence_after();
      const int row = tm * F::BMP + F::BMC * int(rank) + 32 * quarter;
      const uint32_t tbase = tmem_base + (uint32_t(32 * quarter) << 16) + uint32_t(half * (BN / 2));
      uint32_t r[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(tbase + uint32_t(32 * c), r[c]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      // the next tile's MMAs may overwrite it: the loads above have completed (wait::ld), and
      // a release here would also wait for this warp's earlier stores in flight
      if (lane == 0) mbar_arrive_cluster_relaxed(tempty0);
      if (FMT == kNvfp4) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) r[c][i] = __float_as_uint(__uint_as_float(r[c][i]) * alpha);
      }
      constexpr int CW = (EPI == kStoreBf16) ? 32 : 16;  // columns per 64-byte staged row
#pragma unroll
      for (int q = 0; q < (BN / 2) / CW; ++q) {
        if (lane == 0) bulk_wait_group_read<0>();
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
              tma_store_2d_hint(&tmD, buf, col, row, pol_out);
            else
              tma_reduce_add_2d(&tmD, buf, col, row);
          }
          bulk_commit_group();
        }
      }
      acc_phase ^= 1u;
    }
    if (lane == 0) bulk_wait_group_read<0>();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the other may still reach its shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, F::TMEM_COLS);
  }
}

// --------------------------------------------------------------------------- host side

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

template <int FMT, int EPI, int S, bool TSF, bool TILED = false>
gtp_status launch_blockscaled_pair(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &d,
                                   const CUtensorMap &sa, const CUtensorMap &sb, const uint8_t *As, const uint8_t *Bs,
                                   const float *a_amax, const float *b_amax, const Problem &p, int grid,
                                   const gtp::DeviceInfo &dev, cudaStream_t st) {
  using F = BlockScaledPair<FMT, S, TSF, TILED>;
  constexpr auto kernel = gemm_blockscaled_pair_kernel<FMT, EPI, S, TSF, TILED>;
  static std::atomic<uint64_t> configured{0};
  if (gtp_status e = configure(kernel, F::SMEM_TOTAL, configured, dev.device)) return e;
  return gtp::launch_overlapped(kernel, grid, F::THREADS, F::SMEM_TOTAL, st,
                                FMT == kMxfp8 ? "gemm_mxfp8_pair" : "gemm_nvfp4_pair", a, b, d, sa, sb, As, Bs,
                                a_amax, b_amax, p);
}

// The CTA pair unless the output has at most 128 rows (half of every pair tile would be
// empty).  GTP_GEMM_VARIANT=single|pair overrides the choice (read at each call), as for the
// bf16 GEMMs.
bool bs_use_pair(int m_dim) {
  if (const char *v = std::getenv("GTP_GEMM_VARIANT")) {
    if (!std::strcmp(v, "single")) return false;
    if (!std::strcmp(v, "pair")) return true;
  }
  return m_dim > BM;
}

// tiled: the scale arrays are in the tiled layout (gtp_sf_tile); the CTA-pair kernel runs
// whatever the output's height.
template <int FMT, int EPI>
gtp_status run_blockscaled(const uint8_t *Aq, const uint8_t *As, const uint8_t *Bq, const uint8_t *Bs,
                           const float *a_amax, const float *b_amax, void *D, int64_t m_dim, int64_t n_dim,
                           int64_t k_dim, bool allow_split, const gtp::DeviceInfo &dev, cudaStream_t st,
                           bool tiled = false) {
  using F = BlockScaled<FMT>;
  CUtensorMap a, b, d;
  constexpr CU kU8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const int64_t row_bytes = FMT == kMxfp8 ? k_dim : k_dim / 2;
  const int64_t sf_row_bytes = k_dim / F::SF_BLOCK;
  // the pair kernel fetches scale rows by tensor copy when they allow it (16-byte aligned
  // arrays with rows of a multiple of 16 bytes: MXFP8 with K % 512 == 0, every NVFP4
  // shape the entry point accepts), else (MXFP8 only) gathers them with loads
  const bool sf_tma = !tiled && sf_row_bytes % 16 == 0 && gtp::aligned16(As) && gtp::aligned16(Bs);
  const bool pair = tiled || (bs_use_pair(int(m_dim)) && (FMT == kMxfp8 || sf_tma));
  // A boxes are 128 rows either way; B boxes hold the whole 256-row tile, or a CTA's half
  if (gtp_status s = gtp::encode_tmap_2d(&a, kU8, Aq, row_bytes, m_dim, row_bytes, F::BK, BM, kSW128)) return s;
  if (gtp_status s = gtp::encode_tmap_2d(&b, kU8, Bq, row_bytes, n_dim, row_bytes, F::BK, pair ? BN / 2 : BN, kSW128))
    return s;
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
  if (pair) {
    using FP = BlockScaledPair<FMT, 5>;
    // scale rows, 16 bytes (a landing slot's worth) per box
    constexpr CUtensorMapSwizzle kNoSw = CU_TENSOR_MAP_SWIZZLE_NONE;
    CUtensorMap sa = {}, sb = {};
    if (tiled) {  // 512-byte atoms as rows of 128 words; a box is a stage's WORDS atoms
      constexpr CU kU32 = CU_TENSOR_MAP_DATA_TYPE_UINT32;
      const int64_t wrow = k_dim / (4 * F::SF_BLOCK);
      if (gtp_status e = gtp::encode_tmap_2d(&sa, kU32, As, 128, (m_dim + BM - 1) / BM * wrow, 512, 128, F::WORDS,
                                             kNoSw))
        return e;
      if (gtp_status e = gtp::encode_tmap_2d(&sb, kU32, Bs, 128, (n_dim + BM - 1) / BM * wrow, 512, 128, F::WORDS,
                                             kNoSw))
        return e;
    } else if (sf_tma) {
      if (gtp_status e = gtp::encode_tmap_2d(&sa, kU8, As, sf_row_bytes, m_dim, sf_row_bytes, 16, BM, kNoSw))
        return e;
      if (gtp_status e = gtp::encode_tmap_2d(&sb, kU8, Bs, sf_row_bytes, n_dim, sf_row_bytes, 16, BN, kNoSw))
        return e;
    }
    p.tiles_m = int((m_dim + FP::BMP - 1) / FP::BMP);
    p.tiles_n = int((n_dim + BN - 1) / BN);
    p.k_blocks = int(k_dim / FP::K_STAGE);
    const int tiles = p.tiles_m * p.tiles_n, pairs = dev.sm_count / 2;
    p.splits = allow_split ? choose_splits(tiles, p.k_blocks, pairs) : 1;
    p.num_units = tiles * p.splits;
    p.group_m = 2;  // as the bf16 pair GEMM: NVFP4 fc1 (tiled scales) 4.92 -> 5.08 PFLOP/s against 8
    finalize_problem(p);
    const int grid = 2 * std::min(p.num_units, pairs);
    // stage counts measured on the fc1 shapes, PFLOP/s for 4 / 5 / 6 stages: MXFP8 fprop
    // 2.59 / 2.68 / 2.76, dgrad (K 8192) 2.56 / 2.60 / 2.60, wgrad 2.53 / 2.58 / 2.64;
    // NVFP4 runs 4 stages with two landing slots a scale warp (3.52-3.60 against 3.30-3.38
    // for 5 stages with one)
    if constexpr (FMT == kMxfp8) {
      if (tiled)
        return launch_blockscaled_pair<FMT, EPI, 6, true, true>(a, b, d, sa, sb, As, Bs, a_amax, b_amax, p, grid, dev,
                                                                st);
      if (sf_tma)
        return launch_blockscaled_pair<FMT, EPI, 6, true>(a, b, d, sa, sb, As, Bs, a_amax, b_amax, p, grid, dev, st);
      return launch_blockscaled_pair<FMT, EPI, 6, false>(a, b, d, sa, sb, As, Bs, a_amax, b_amax, p, grid, dev, st);
    } else {  // NVFP4 scale arrays are always 16-byte aligned with 16-byte multiple rows
      if (tiled)
        return launch_blockscaled_pair<FMT, EPI, 5, true, true>(a, b, d, sa, sb, As, Bs, a_amax, b_amax, p, grid, dev,
                                                                st);
      return launch_blockscaled_pair<FMT, EPI, 5, true>(a, b, d, sa, sb, As, Bs, a_amax, b_amax, p, grid, dev, st);
    }
  }
  p.tiles_m = int((m_dim + BM - 1) / BM);
  p.tiles_n = int((n_dim + BN - 1) / BN);
  p.k_blocks = int(k_dim / F::K_STAGE);
  const int tiles = p.tiles_m * p.tiles_n;
  p.splits = allow_split ? choose_splits(tiles, p.k_blocks, dev.sm_count) : 1;
  p.num_units = tiles * p.splits;
  p.group_m = 16;
  finalize_problem(p);
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

namespace {
// main_grad[N, K] += dq(dYtq)[N, M] · dq(Xtq)[K, M]^T: contraction M
gtp_status wgrad_mxfp8(const uint8_t *dYtq, const uint8_t *dYts, const uint8_t *Xtq, const uint8_t *Xts,
                       float *grad_data, int64_t grad_offset, int64_t grad_numel_total, int64_t M, int64_t N,
                       int64_t K, bool tiled, gtp_stream stream) {
  if (grad_offset < 0 || grad_numel_total < 0) return gtp::fail(GTP_E_ARG, "negative offset or size");
  if (N * K > grad_numel_total - grad_offset)
    return gtp::fail(GTP_E_RANGE, "view [%lld, +%lld) exceeds the grad buffer (%lld)", (long long)grad_offset,
                     (long long)(N * K), (long long)grad_numel_total);
  if (grad_offset % 4) return gtp::fail(GTP_E_ALIGN, "grad_offset must be a multiple of 4 elements");
  float *view = grad_data ? grad_data + grad_offset : nullptr;
  if (gtp_status s = check_mxfp8(dYtq, dYts, Xtq, Xts, view, N, K, M, 4)) return s;
  if (M == 0 || N == 0 || K == 0) return GTP_OK;
  if (tiled && (!gtp::aligned16(dYts) || !gtp::aligned16(Xts)))
    return gtp::fail(GTP_E_ALIGN, "tiled scale pointers must be 16-byte aligned");
  gtp::DeviceInfo dev;
  if (gtp_status s = gtp::require_sm103(&dev)) return s;
  return run_blockscaled<kMxfp8, kReduceAddF32>(dYtq, dYts, Xtq, Xts, nullptr, nullptr, view, N, K, M, true, dev,
                                                gtp::as_stream(stream), tiled);
}

// dX[M, K] = dq(dYq)[M, N] · dq(Wtq)[K, N]^T: contraction N, output columns K
gtp_status dgrad_mxfp8(const uint8_t *dYq, const uint8_t *dYs, const uint8_t *Wtq, const uint8_t *Wts, void *dX,
                       int64_t M, int64_t N, int64_t K, bool tiled, gtp_stream stream) {
  if (gtp_status s = check_mxfp8(dYq, dYs, Wtq, Wts, dX, M, K, N, 2)) return s;
  if (M == 0 || K == 0) return GTP_OK;
  if (tiled && N > 0 && (!gtp::aligned16(dYs) || !gtp::aligned16(Wts)))
    return gtp::fail(GTP_E_ALIGN, "tiled scale pointers must be 16-byte aligned");
  gtp::DeviceInfo dev;
  if (gtp_status s = gtp::require_sm103(&dev)) return s;
  cudaStream_t st = gtp::as_stream(stream);
  if (N == 0) return gtp::launch_zero_bytes(dX, M * K * 2, st, dev.sm_count);
  return run_blockscaled<kMxfp8, kStoreBf16>(dYq, dYs, Wtq, Wts, nullptr, nullptr, dX, M, K, N, false, dev, st, tiled);
}
}  // namespace

extern "C" gtp_status gtp_linear_dgrad_mxfp8(const uint8_t *dYq, const uint8_t *dYs, const uint8_t *Wtq,
                                             const uint8_t *Wts, void *dX, int64_t M, int64_t N, int64_t K,
                                             gtp_stream stream) {
  gtp::clear_error();
  return dgrad_mxfp8(dYq, dYs, Wtq, Wts, dX, M, N, K, false, stream);
}

extern "C" gtp_status gtp_linear_wgrad_accum_mxfp8(const uint8_t *dYtq, const uint8_t *dYts, const uint8_t *Xtq,
                                                   const uint8_t *Xts, float *grad_data, int64_t grad_offset,
                                                   int64_t grad_numel_total, int64_t M, int64_t N, int64_t K,
                                                   gtp_stream stream) {
  gtp::clear_error();
  return wgrad_mxfp8(dYtq, dYts, Xtq, Xts, grad_data, grad_offset, grad_numel_total, M, N, K, false, stream);
}

extern "C" gtp_status gtp_linear_wgrad_accum_mxfp8_tiled(const uint8_t *dYtq, const uint8_t *dYts_tiled,
                                                         const uint8_t *Xtq, const uint8_t *Xts_tiled,
                                                         float *grad_data, int64_t grad_offset,
                                                         int64_t grad_numel_total, int64_t M, int64_t N, int64_t K,
                                                         gtp_stream stream) {
  gtp::clear_error();
  return wgrad_mxfp8(dYtq, dYts_tiled, Xtq, Xts_tiled, grad_data, grad_offset, grad_numel_total, M, N, K, true,
                     stream);
}

extern "C" gtp_status gtp_linear_dgrad_mxfp8_tiled(const uint8_t *dYq, const uint8_t *dYs_tiled, const uint8_t *Wtq,
                                                   const uint8_t *Wts_tiled, void *dX, int64_t M, int64_t N,
                                                   int64_t K, gtp_stream stream) {
  gtp::clear_error();
  return dgrad_mxfp8(dYq, dYs_tiled, Wtq, Wts_tiled, dX, M, N, K, true, stream);
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

extern "C" gtp_status gtp_linear_fprop_nvfp4_tiled(const uint8_t *Xq, const uint8_t *Xs_tiled, const float *x_amax,
                                                   const uint8_t *Wq, const uint8_t *Ws_tiled, const float *w_amax,
                                                   void *Y, int64_t M, int64_t N, int64_t K, gtp_stream stream) {
  gtp::clear_error();
  if (gtp_status s = check_mxfp8(Xq, Xs_tiled, Wq, Ws_tiled, Y, M, N, K, 2, BlockScaled<kNvfp4>::K_STAGE)) return s;
  if (M == 0 || N == 0) return GTP_OK;
  if (K > 0 && (!x_amax || !w_amax)) return gtp::fail(GTP_E_ARG, "null amax");
  if ((reinterpret_cast<uintptr_t>(x_amax) | reinterpret_cast<uintptr_t>(w_amax)) & 3u)
    return gtp::fail(GTP_E_ALIGN, "amax pointers must be 4-byte aligned");
  if (K > 0 && (!gtp::aligned16(Xs_tiled) || !gtp::aligned16(Ws_tiled)))
    return gtp::fail(GTP_E_ALIGN, "tiled scale pointers must be 16-byte aligned");
  gtp::DeviceInfo dev;
  if (gtp_status s = gtp::require_sm103(&dev)) return s;
  cudaStream_t st = gtp::as_stream(stream);
  if (K == 0) return gtp::launch_zero_bytes(Y, M * N * 2, st, dev.sm_count);
  return run_blockscaled<kNvfp4, kStoreBf16>(Xq, Xs_tiled, Wq, Ws_tiled, x_amax, w_amax, Y, M, N, K, false, dev, st,
                                             true);
}

extern "C" gtp_status gtp_linear_fprop_mxfp8_tiled(const uint8_t *Xq, const uint8_t *Xs_tiled, const uint8_t *Wq,
                                                   const uint8_t *Ws_tiled, void *Y, int64_t M, int64_t N, int64_t K,
                                                   gtp_stream stream) {
  gtp::clear_error();
  if (gtp_status s = check_mxfp8(Xq, Xs_tiled, Wq, Ws_tiled, Y, M, N, K, 2)) return s;
  if (M == 0 || N == 0) return GTP_OK;
  if (K > 0 && (!gtp::aligned16(Xs_tiled) || !gtp::aligned16(Ws_tiled)))
    return gtp::fail(GTP_E_ALIGN, "tiled scale pointers must be 16-byte aligned");
  gtp::DeviceInfo dev;
  if (gtp_status s = gtp::require_sm103(&dev)) return s;
  cudaStream_t st = gtp::as_stream(stream);
  if (K == 0) return gtp::launch_zero_bytes(Y, M * N * 2, st, dev.sm_count);
  return run_blockscaled<kMxfp8, kStoreBf16>(Xq, Xs_tiled, Wq, Ws_tiled, nullptr, nullptr, Y, M, N, K, false, dev, st,
                                             true);
}

namespace gtp {
gtp_status blockscaled_wait_word(unsigned int *v, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(v, g_gtp_wait_timeouts, sizeof(*v));
  if (e == cudaSuccess && reset) {
    const unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_gtp_wait_timeouts, &z, sizeof(z));
  }
  if (e != cudaSuccess) return fail(GTP_E_CUDA, "reading the wait-timeout word: %s", cudaGetErrorString(e));
  return GTP_OK;
}
}  // namespace gtp
