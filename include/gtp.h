/*
 * gtp.h - C ABI of the GB300 (sm_103a) hot path of a tensor-parallel linear layer and
 * its flat param/grad buffer.
 *
 * Pages cited (title, section):
 *   [LIN] "01 · ColumnParallelLinear / RowParallelLinear and the core autograd"
 *         (llm-infra-atlas) - forward §4.1, backward §4.2.
 *   [BUF] "05 · grad/param buffer: contiguous buffer data structures and read/write
 *         loop" (llm-infra-atlas) - BufferKey §3, layout §4.1-§4.3, mounting §5,
 *         start_grad_sync §6.3, the ZeRO-1 param loop §6.5, zero_grad_buffer §6.6.
 *   [MLM] "Megatron-LM architecture and source guide" (arganzheng.life) - run.sh
 *         hyper-parameters §4, DistributedOptimizer step §6.4.
 *   [GTP] "Generalized Tensor Parallelism (GTP)" (Megatron-Core developer guide) -
 *         native MXFP8 weights, §1.3 and its "Communication volume breakdown" table.
 *
 * Conventions for every entry point:
 *   - Pointers named as device pointers must point to device memory of the current
 *     CUDA device; pointers named as host pointers to host memory.  The caller owns
 *     all memory; no entry point allocates, frees or keeps a pointer after it returns.
 *   - Matrices are dense, row-major and contiguous.  Notation: M tokens, N out-features
 *     and K in-features of one TP shard; X [M,K], W [N,K], Y and dY [M,N], dX [M,K],
 *     main_grad [N,K].
 *   - GPU work is enqueued asynchronously on `stream` (a cudaStream_t passed as a
 *     void*; NULL is the legacy default stream) and the call returns without
 *     synchronising.
 *   - Argument errors are detected on the host and returned before anything is
 *     launched; nothing is written in that case.  A failed launch returns
 *     GTP_E_CUDA.  gtp_last_error() gives a message for the calling thread.  No entry
 *     point aborts, throws or falls back to another implementation.
 *
 * Environment switches (read at each call; unset is the default the measurements chose).
 * They change how a result is computed, never what it is, beyond the fp32 summation
 * order of split wgrad contractions; they exist for tests and timing comparisons:
 *   GTP_GEMM_VARIANT=single|pair  the bf16 GEMMs' one-CTA or CTA-pair kernel for every
 *                                 shape (default: the pair kernel above 128 output rows);
 *   GTP_GEMM_SCHED=dynamic        the CTA-pair kernel's cluster-launch-control schedule
 *                                 instead of the static round-robin;
 *   GTP_GEMM_TAIL=full            whole tiles in the last partial wave (default: half-
 *                                 width tail units where they fit);
 *   GTP_GEMM_L2HINT=off           operand loads without the L2 evict_first/last policies;
 *   GTP_GROUP_SPLITS=<n>          a fixed split count for the splittable wgrad products of a
 *                                 grouped launch (default: the planner's choice; read when
 *                                 the process first plans a group of that shape);
 *   GTP_MXCOL_VARIANT=strip       the strip kernel for every columnwise MXFP8 quantization
 *                                 (default: the warp-tile kernel where rows are 16-byte);
 *   GTP_NO_LAUNCH_OVERLAP=<any>   launches without programmatic dependent launch.
 */
#ifndef GTP_H_
#define GTP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GTP_OK = 0,
  GTP_E_ARG = 1,        /* null pointer, negative size, bad flag or hyper-parameter   */
  GTP_E_SHAPE = 2,      /* a dimension the kernel cannot take (e.g. K % 32 for MX)     */
  GTP_E_ALIGN = 3,      /* pointer / offset / row stride not 16-byte aligned           */
  GTP_E_DTYPE = 4,      /* dtype not supported by this entry point                     */
  GTP_E_RANGE = 5,      /* a view or bucket range outside its buffer, or overlapping   */
  GTP_E_CAPACITY = 6,   /* an output array too small / more buckets than supported     */
  GTP_E_CUDA = 7,       /* a CUDA runtime or driver call failed                        */
  GTP_E_DEVICE = 8      /* the current device is not an sm_103 GPU                     */
} gtp_status;

typedef enum { GTP_F32 = 0, GTP_BF16 = 1, GTP_F16 = 2, GTP_U8 = 3 } gtp_dtype;

typedef void *gtp_stream; /* cudaStream_t */

/* Message describing the last error returned on the calling thread ("" if none). */
const char *gtp_last_error(void);

/* ------------------------------------------------------------------------ GEMMs
 * One TP shard of LinearWithGradAccumulationAndAsyncCommunication ([LIN] §4.1, §4.2).
 * All three run on the 5th-generation tensor cores (tcgen05, fp32 accumulation in
 * tensor memory) with operands staged by TMA.  `dt` must be GTP_BF16.
 * Requirements: M, N, K >= 0; every base pointer 16-byte aligned; every row stride a
 * multiple of 16 bytes (K % 8 == 0 and N % 8 == 0 for bf16 rows).
 */

/* Y[M,N] = X[M,K] · W[N,K]^T  ([LIN] §4.1 "output = torch.matmul(total_input,
 * weight.t())").  fp32 accumulation, one round-to-nearest-even to bf16.  K == 0
 * writes zeros.  X, W, Y: device pointers. */
gtp_status gtp_linear_fprop(const void *X, const void *W, void *Y, int64_t M, int64_t N,
                            int64_t K, gtp_dtype dt, gtp_stream stream);

/* dX[M,K] = dY[M,N] · W[N,K]  ([LIN] §4.2 dgrad "grad_output.matmul(weight)").
 * fp32 accumulation, RNE to bf16.  N == 0 writes zeros.  dY, W, dX: device pointers. */
gtp_status gtp_linear_dgrad(const void *dY, const void *W, void *dX, int64_t M, int64_t N,
                            int64_t K, gtp_dtype dt, gtp_stream stream);

/* main_grad[N,K] += dY[M,N]^T · X[M,K] in fp32, where main_grad is the view
 * grad_data[grad_offset : grad_offset + N*K] of the flat fp32 grad buffer
 * ([LIN] §4.2 wgrad with gradient_accumulation_fusion; [BUF] §5
 * "param.main_grad = grad_data[s:e].view(shape)").  Never zeroes main_grad (that is
 * gtp_buffer_zero's job, [BUF] §6.6); microbatch accumulation is repeated calls.
 * The fp32 sum of the tile partials is formed by in-memory fp32 additions, so the
 * rounding order (not the result's accuracy) can differ between runs.
 * The view may start at any element ([BUF] §4.2: the default, unpadded layout places a
 * parameter right after the previous one): a view whose start is 16-byte aligned (every
 * distributed-optimizer view: starts are multiples of 64 elements) is accumulated by TMA
 * fp32 reduce-adds, any other by fp32 atomic adds from registers (slower).
 * Extra requirements: grad_data 4-byte aligned, grad_offset + N*K <= grad_numel_total
 * (else GTP_E_RANGE).  dY, X (16-byte aligned), grad_data: device pointers. */
gtp_status gtp_linear_wgrad_accum(const void *dY, const void *X, float *grad_data,
                                  int64_t grad_offset, int64_t grad_numel_total, int64_t M,
                                  int64_t N, int64_t K, gtp_dtype dt, gtp_stream stream);

/* gtp_linear_wgrad_accum with a bit-reproducible result: the contraction over M is never
 * split, so each element of main_grad receives exactly one fp32 addition per call, of a
 * sum formed on one CTA pair in a fixed order.  Two identical sequences of calls give
 * bit-identical buffers (Megatron's fused fp32 accumulate, [LIN] §4.2
 * wgrad_gemm_accum_fp32, is likewise deterministic).  Same arguments, requirements and
 * errors; it gives up the split that fills the GPU on shapes with few output tiles. */
gtp_status gtp_linear_wgrad_accum_deterministic(const void *dY, const void *X,
                                                float *grad_data, int64_t grad_offset,
                                                int64_t grad_numel_total, int64_t M, int64_t N,
                                                int64_t K, gtp_dtype dt, gtp_stream stream);

/* The same accumulate into a bf16 grad buffer (grad_reduce_in_fp32 off: [BUF] §3, the
 * BufferKey's grad_dtype is the parameter's bf16; the accumulation is still computed in
 * fp32): main_grad[N,K] = RNE_bf16(main_grad + dY^T · X), one rounding of the fp32 sum a
 * call, where main_grad is the view grad_data[grad_offset : grad_offset + N*K] of a bf16
 * buffer.  The contraction is never split (each element is read, summed and written by
 * one CTA pair), so the result is bit-reproducible.  The view may start at any element;
 * grad_data: device, 2-byte aligned; other arguments and errors as gtp_linear_wgrad_accum. */
gtp_status gtp_linear_wgrad_accum_bf16(const void *dY, const void *X, void *grad_data,
                                       int64_t grad_offset, int64_t grad_numel_total, int64_t M,
                                       int64_t N, int64_t K, gtp_dtype dt, gtp_stream stream);

/* ---------------------------------------------------------------- grouped launches
 * Several independent products in ONE launch of the CTA-pair kernel: their output tiles
 * (and, for wgrad, contraction ranges) form one list that the 76 CTA pairs take in turn,
 * so the launch's start-up, its last partial wave and its last epilogue are paid once for
 * the group, and one product's short last wave fills with the next product's tiles.  Each
 * product computes exactly what its single entry point computes, with the same arguments,
 * requirements and errors; the results are the same up to the fp32 summation order of
 * split wgrad contractions (none with GTP_GEMM_DETERMINISTIC).
 * The products must be independent: no output may overlap an input or another output
 * (GTP_E_ARG, found before anything is launched); inputs may be shared, and two fp32
 * WGRAD_ACCUM views of one buffer may overlap (their fp32 additions commute, in either
 * order: such a group is not bit-reproducible, even with GTP_GEMM_DETERMINISTIC).
 */
typedef enum { GTP_GEMM_FPROP = 0, GTP_GEMM_DGRAD = 1, GTP_GEMM_WGRAD_ACCUM = 2 } gtp_gemm_kind;

typedef struct {
  int32_t kind;               /* gtp_gemm_kind                                             */
  int32_t dtype;              /* gtp_dtype of the operands: GTP_BF16                        */
  const void *a;              /* FPROP: X [M,K];  DGRAD: dY [M,N];  WGRAD_ACCUM: dY [M,N]   */
  const void *b;              /* FPROP: W [N,K];  DGRAD: W [N,K];   WGRAD_ACCUM: X [M,K]    */
  void *out;                  /* FPROP: Y [M,N];  DGRAD: dX [M,K];  WGRAD_ACCUM: grad_data */
  int64_t M, N, K;            /* as for the single entry points                             */
  int64_t grad_offset;        /* WGRAD_ACCUM: first element of the main_grad view           */
  int64_t grad_numel_total;   /* WGRAD_ACCUM: elements of grad_data                          */
  int32_t grad_dtype;         /* WGRAD_ACCUM: GTP_F32 (gtp_linear_wgrad_accum's arithmetic)  */
                              /*   or GTP_BF16 (gtp_linear_wgrad_accum_bf16's, never split)  */
  int32_t reserved;           /* must be 0                                                   */
} gtp_gemm_desc;

enum { GTP_GEMM_DETERMINISTIC = 1 }; /* flags: never split a wgrad contraction */

/* Runs descs[0..n) (0 <= n <= 4; host array of device pointers) on `stream`.  Every
 * descriptor is validated before anything is launched.  Products with at most 128 output
 * rows (the single-CTA kernel) and empty contractions (zeros) are launched on their own,
 * before the group.  reserved must be 0 (GTP_E_ARG otherwise). */
gtp_status gtp_linear_grouped(const gtp_gemm_desc *descs, int32_t n, int32_t flags,
                              gtp_stream stream);

/* The backward of one linear shard ([LIN] §4.2: dgrad and the fused wgrad accumulate of
 * LinearWithGradAccumulationAndAsyncCommunication, whose TP collectives are out of scope
 * on one GPU) as one grouped launch: dX[M,K] = dY[M,N] · W[N,K] and
 * main_grad[N,K] += dY^T · X[M,K] into grad_data[grad_offset : grad_offset + N*K].
 * Arguments and errors as gtp_linear_dgrad and gtp_linear_wgrad_accum; flags as
 * gtp_linear_grouped. */
gtp_status gtp_linear_backward(const void *dY, const void *X, const void *W, void *dX,
                               float *grad_data, int64_t grad_offset, int64_t grad_numel_total,
                               int64_t M, int64_t N, int64_t K, gtp_dtype dt, int32_t flags,
                               gtp_stream stream);

/* ------------------------------------------------------------------ buffer layout
 * Host-only: computes the layout of the flat param/grad buffers; launches nothing and
 * needs no GPU.  Follows [BUF] §3 (BufferKey grouping, keys in order of first
 * appearance), §4.1 (reverse model order), §4.2 (dist-opt: param starts rounded up to
 * 64 elements, bucket ends to lcm(dp,128) or lcm(dp,128,2^16), a shared embedding in
 * a bucket of its own; default mode: no padding), §4.3 (cut after the parameter whose
 * end reaches bucket_size elements from the bucket start) and §5 (param_index_map).
 */
typedef struct {
  int64_t numel;               /* elements of the parameter, > 0                       */
  int32_t dtype;               /* gtp_dtype of the parameter (F32, BF16 or F16)        */
  int32_t quantized_storage;   /* 1: FP8/NVFP4 parameter, buffer key dtype is uint8    */
  int32_t is_expert_parallel;  /* 1: not param.allreduce                               */
  int32_t is_layer_wise;       /* 1: managed by the layer-wise optimizer               */
  int32_t is_shared_embedding; /* 1: tied embedding (own bucket in dist-opt mode)      */
  int32_t reserved;            /* must be 0                                            */
} gtp_param_desc;

typedef struct {
  int64_t bucket_size;                     /* elements; <= 0 means one bucket           */
  int32_t dp_size;                         /* >= 1                                     */
  int32_t use_distributed_optimizer;       /* 0: no padding at all                      */
  int32_t pad_buckets_for_high_nccl_busbw; /* 1: bucket ends to lcm(dp,128,65536)       */
  int32_t grad_reduce_in_fp32;             /* 1: grad dtype fp32, else the param dtype  */
} gtp_layout_config;

typedef struct {
  int64_t start, end;                   /* [start, end) in its buffer (param_index_map) */
  int64_t start_in_bucket, end_in_bucket; /* param_to_index of its bucket               */
  int32_t bucket_id;                    /* global bucket index                          */
  int32_t buffer_id;
} gtp_param_index;

typedef struct {
  int64_t offset;         /* first element of the bucket in its buffer                  */
  int64_t numel_unpadded; /* up to the end of its last parameter                        */
  int64_t numel;          /* including the end padding                                  */
  int32_t buffer_id;
  int32_t num_params;
} gtp_bucket_desc;

typedef struct {
  int64_t numel;          /* total elements incl. padding (grad_data / param_data size) */
  int32_t param_dtype;    /* BufferKey.param_dtype (GTP_U8 for quantized storage)       */
  int32_t grad_dtype;     /* BufferKey.grad_dtype                                       */
  int32_t is_expert_parallel;
  int32_t is_layer_wise;
  int32_t first_bucket;   /* this buffer's buckets are [first_bucket, +num_buckets)    */
  int32_t num_buckets;
} gtp_buffer_desc;

/* params[n_params] (host, MODEL order) -> index[n_params] (host, may be NULL),
 * buffers[*n_buffers] and buckets[*n_buckets] (host).  On entry *n_buffers and
 * *n_buckets hold the capacities of `buffers` / `buckets` (0 with NULL arrays to query);
 * on return they hold the counts.  Too small a capacity returns GTP_E_CAPACITY after
 * writing the counts (and `index` if given), so a first call with NULL arrays sizes
 * the second.  Buckets are numbered buffer by buffer, each in offset order. */
gtp_status gtp_buffer_layout(const gtp_param_desc *params, int32_t n_params,
                             const gtp_layout_config *cfg, gtp_param_index *index,
                             gtp_buffer_desc *buffers, int32_t *n_buffers,
                             gtp_bucket_desc *buckets, int32_t *n_buckets);

/* Distributed-optimizer range map of one dp rank ([BUF] §6.5, [MLM] §6.4): every bucket
 * of a buffer is cut into dp equal element shards, rank r owning the r-th, regardless of
 * parameter boundaries; for each parameter that overlaps rank r's shard of its bucket the
 * overlap is given in four frames (Megatron's gbuf_world, gbuf_world_in_bucket,
 * gbuf_local and param ranges).  Host-only. */
typedef struct {
  int32_t param;          /* index into the parameter list given to gtp_buffer_layout     */
  int32_t bucket_id;
  int64_t world_start;    /* overlap in the buffer: [world_start, world_end)              */
  int64_t world_end;
  int64_t bucket_start;   /* world_start - bucket offset                                  */
  int64_t local_start;    /* world_start - start of this rank's shard of the bucket      */
  int64_t param_start;    /* world_start - parameter start (offset inside the parameter) */
} gtp_shard_range;

/* index[n_params] and buckets[n_buckets]: host arrays as written by gtp_buffer_layout.
 * Ranges of buffer `buffer_id` for rank dp_rank of dp_size, ordered by bucket then by
 * position.  Two-call protocol on *n_out (capacity in, count out; NULL `out` to query).
 * Every bucket of the buffer must divide by dp_size (GTP_E_SHAPE otherwise, which the
 * dist-opt layout guarantees). */
gtp_status gtp_shard_param_ranges(const gtp_param_index *index, int32_t n_params,
                                  const gtp_bucket_desc *buckets, int32_t n_buckets,
                                  int32_t buffer_id, int32_t dp_size, int32_t dp_rank,
                                  gtp_shard_range *out, int32_t *n_out);

/* ------------------------------------------------------------- flat-buffer sweep */

/* data[0:numel] = 0 over the whole buffer including padding ([BUF] §6.6
 * zero_grad_buffer -> grad_data.zero_()).  dt: F32, BF16, F16 or U8 (element size
 * only).  data: device pointer, 16-byte aligned. */
gtp_status gtp_buffer_zero(void *data, gtp_dtype dt, int64_t numel, gtp_stream stream);

/* grad_data[b.offset : b.offset + b.numel] *= factors[b] for every bucket b, fp32, in
 * place ([BUF] §6.3: start_grad_sync pre-multiplies by gradient_scaling_factor).
 * buckets and factors: host arrays of n_buckets entries whose ranges
 * lie inside [0, grad_numel) and do not overlap (at most 512 buckets).  grad_data: device, 16-byte aligned. */
gtp_status gtp_bucket_scale(float *grad_data, int64_t grad_numel, const gtp_bucket_desc *buckets,
                            const float *factors, int32_t n_buckets, gtp_stream stream);

typedef struct {
  float lr, beta1, beta2, eps, weight_decay; /* AdamW; weight_decay 0 gives Adam         */
  int32_t zero_grad_after;                   /* 1: write grad_data = 0 after reading it  */
  int64_t step;                              /* 1-based step count t                     */
  const float *grad_scale;                   /* device pointer to one float multiplying
                                                every scaled gradient (the clip
                                                coefficient of gtp_grad_norm); NULL = 1  */
} gtp_adam_hparams;

/* One fused HBM sweep over the flat buffer, per element i in [0, numel):
 *   g   = (grad_data[i] * factor(bucket of i)) * grad_scale  ([BUF] §6.3 scaling, clip)
 *   m   = b1 m + (1-b1) g;   v = b2 v + (1-b2) g^2      (Adam, [BUF] §6.5 ②)
 *   p   = p (1 - lr wd) - (lr / (1-b1^t)) m / (sqrt(v)/sqrt(1-b2^t) + eps)
 *   param_data[i] = bf16_rne(p)                          ([BUF] §6.5 ③, [MLM] §6.4)
 *   grad_data[i]  = 0 if zero_grad_after                 ([BUF] §6.6, moved here)
 * master (p), exp_avg (m), exp_avg_sq (v): fp32; param_data: bf16.  All device
 * pointers, 16-byte aligned, numel elements each; no two of the five arrays may share a
 * byte (GTP_E_ARG, before any launch).  Elements outside every bucket use
 * factor 1.  buckets/factors: host arrays as for gtp_bucket_scale (may be NULL with
 * n_buckets 0).  h: host pointer. */
gtp_status gtp_adam_step_flat(float *grad_data, float *master, float *exp_avg,
                              float *exp_avg_sq, void *param_data, int64_t numel,
                              const gtp_bucket_desc *buckets, const float *factors,
                              int32_t n_buckets, const gtp_adam_hparams *h, gtp_stream stream);

/* gtp_adam_step_flat for a bf16 grad buffer (grad_reduce_in_fp32 off, [BUF] §3 BufferKey
 * grad_dtype bf16): step ① of [BUF] §6.5 (shard_main_param.grad =
 * shard_model_grad.float()) is then a real conversion, done in registers (exact); the
 * rest is unchanged, and the zeroing writes bf16 zeros.  30 bytes of HBM traffic an
 * element instead of 34.  grad_data: device, 16-byte aligned, numel bf16 elements;
 * everything else as gtp_adam_step_flat. */
gtp_status gtp_adam_step_flat_bf16_grad(void *grad_data, float *master, float *exp_avg,
                                        float *exp_avg_sq, void *param_data, int64_t numel,
                                        const gtp_bucket_desc *buckets, const float *factors,
                                        int32_t n_buckets, const gtp_adam_hparams *h,
                                        gtp_stream stream);

/* The same sweep for a buffer of native MXFP8 parameters ([GTP] §1.3: the optimizer
 * writes the FP8 weight from the fp32 master once per step; [BUF] §3: such a buffer's
 * param_data has the storage dtype uint8).  Instead of the bf16 cast, every aligned block
 * of 32 elements j in [32q, 32q+32) of the updated master is written as
 *   param_e8m0[q]  = E8M0 scale byte, 2^(floor(log2 amax) - 8) clamped (OCP MX rule)
 *   param_e4m3[j]  = RNE E4M3 of p_j / scale, saturating at +-448
 * (a block with NaN/Inf: scale 0xFF, codes 0x7F).  A weight [N, K] at a buffer offset
 * that is a multiple of 32, with K % 32 == 0, thus has its rowwise MXFP8 view at
 * param_e4m3 + offset ([N, K]) and param_e8m0 + offset / 32 ([N, K/32]), ready for
 * gtp_linear_fprop_mxfp8.  numel must be a multiple of 32 (GTP_E_SHAPE); param_e4m3:
 * device, numel bytes, 16-byte aligned; param_e8m0: device, numel / 32 bytes, 4-byte
 * aligned (GTP_E_ALIGN otherwise).  Other
 * arguments and errors as gtp_adam_step_flat. */
gtp_status gtp_adam_step_flat_mxfp8(float *grad_data, float *master, float *exp_avg,
                                    float *exp_avg_sq, uint8_t *param_e4m3, uint8_t *param_e8m0,
                                    int64_t numel, const gtp_bucket_desc *buckets,
                                    const float *factors, int32_t n_buckets,
                                    const gtp_adam_hparams *h, gtp_stream stream);

/* ------------------------------------------------------- gradient norm and clipping
 * [BUF] §6.3: before the collective, start_grad_sync can compute each bucket's gradient
 * L2 norm and reject NaN/Inf (fatal) or abnormally large (non-fatal) gradients; [MLM] §4
 * trains with --clip-grad 1.0.  For the scaled gradient v = factor_b * g of every bucket:
 *   sumsq[b]     = sum of v^2 over bucket b (fp64 result, fp32 squares),
 *   nonfinite[b] = number of non-finite v in bucket b,
 *   *total_norm  = sqrt(sum_b sumsq[b]),
 *   *clip_coef   = min(1, max_norm / (*total_norm + 1e-6)), or 1 when max_norm == 0.
 * A non-finite gradient makes the norm non-finite; the caller reads nonfinite[] and skips
 * the step.  Deterministic: no atomics, a fixed reduction order.  Two launches; the
 * coefficient stays on the device for gtp_adam_hparams.grad_scale.
 * buckets/factors: host arrays (1 to 512 buckets, inside [0, numel)); grad_data: device,
 * 16-byte aligned; sumsq[n_buckets], nonfinite[n_buckets], total_norm, clip_coef: device.
 * workspace: device scratch of at least gtp_grad_norm_workspace_bytes(buckets, n)
 * bytes (16-byte aligned), owned by the caller; its contents are not needed afterwards.
 * Returns GTP_E_CAPACITY when the workspace is too small. */
size_t gtp_grad_norm_workspace_bytes(const gtp_bucket_desc *buckets, int32_t n_buckets);

gtp_status gtp_grad_norm(const float *grad_data, int64_t numel, const gtp_bucket_desc *buckets,
                         const float *factors, int32_t n_buckets, float max_norm, void *workspace,
                         size_t workspace_bytes, double *sumsq, uint32_t *nonfinite,
                         float *total_norm, float *clip_coef, gtp_stream stream);

/* gtp_grad_norm without a workspace argument, for callers that cannot allocate device
 * memory where they need the norm: code under a fixed memory budget whose allocator must
 * not be re-entered (an out-of-memory handler of a caching allocator, a full arena), or a
 * plain C caller with no device allocator of its own.  The pages have no counterpart;
 * this is a convenience of this library.
 * The chunk partials live in a 1 MiB array inside the library's device image (every GPU
 * that loads the library keeps it until the process exits), which bounds the input to
 * 65536 chunks of 65536 elements (about 4.29e9 elements, fewer when buckets end
 * mid-chunk); a larger input returns GTP_E_CAPACITY and needs gtp_grad_norm.
 * The first call on a device looks up that array's device address (once per device, with
 * that device current); make that first call before any stream capture.
 * Every call, on every stream, shares the one array: calls that overlap on the GPU race
 * and produce wrong results, so serialise them (one stream, or events).  Nothing in the
 * array has to start at zero: each call writes every partial it reads.
 * Arguments, outputs and errors as gtp_grad_norm; it calls no allocation routine. */
gtp_status gtp_grad_norm_noalloc(const float *grad_data, int64_t numel,
                                 const gtp_bucket_desc *buckets, const float *factors,
                                 int32_t n_buckets, float max_norm, double *sumsq,
                                 uint32_t *nonfinite, float *total_norm, float *clip_coef,
                                 gtp_stream stream);

/* ----------------------------------------------------------------------- MXFP8
 * Native MXFP8 weights ([GTP] §1.3): E4M3 elements plus one E8M0 scale byte per block
 * of 32 consecutive elements of a row ("Block 32", scale 1/32 B/elem).  The scale of
 * a block is 2^(floor(log2(amax)) - 8) clamped to [2^-127, 2^127] (OCP MX rule), each
 * element RNE(x / scale) saturated to +-448.  amax == 0 gives scale byte 0 and zero
 * elements; a block holding NaN or Inf gives scale 0xFF and elements 0x7F.
 */

/* src[rows,cols] (F32 or BF16) -> e4m3[rows,cols], e8m0[rows, cols/32].
 * cols % 32 == 0 (else GTP_E_SHAPE).  All device pointers; src 16-byte aligned. */
gtp_status gtp_mxfp8_quantize_rowwise(const void *src, gtp_dtype src_dt, int64_t rows,
                                      int64_t cols, uint8_t *e4m3, uint8_t *e8m0,
                                      gtp_stream stream);

/* The columnwise (backward) view ([GTP] §1.3: "the rowwise (fwd) / columnwise (bwd)
 * view"): blocks of 32 consecutive ROWS of each column, stored transposed so that each
 * column becomes a row: e4m3_t[cols, rows], e8m0_t[cols, rows/32] - the rowwise
 * quantization of src^T.  rows % 32 == 0.  src (F32 or BF16): device, element-aligned;
 * e4m3_t: device, 16-byte aligned; e8m0_t: device. */
gtp_status gtp_mxfp8_quantize_columnwise(const void *src, gtp_dtype src_dt, int64_t rows,
                                         int64_t cols, uint8_t *e4m3_t, uint8_t *e8m0_t,
                                         gtp_stream stream);

/* The same view with its scales in the tiled layout (gtp_sf_tile's order of the
 * [cols, rows / 32] array): e8m0_t_tiled holds gtp_sf_tiled_bytes(cols, rows / 32) bytes,
 * 16-byte aligned (GTP_E_ALIGN otherwise); its padding bytes are left unwritten.  This is
 * what gtp_linear_dgrad_mxfp8_tiled and gtp_linear_wgrad_accum_mxfp8_tiled read. */
gtp_status gtp_mxfp8_quantize_columnwise_tiled(const void *src, gtp_dtype src_dt, int64_t rows,
                                               int64_t cols, uint8_t *e4m3_t,
                                               uint8_t *e8m0_t_tiled, gtp_stream stream);

/* One matrix of gtp_mxfp8_quantize_columnwise_group: the arguments of
 * gtp_mxfp8_quantize_columnwise (tiled_scales 0) or gtp_mxfp8_quantize_columnwise_tiled
 * (tiled_scales 1), with the same meaning and rules. */
typedef struct {
  const void *src;       /* [rows, cols] F32 or BF16, device */
  uint8_t *e4m3_t;       /* [cols, rows], device, 16-byte aligned */
  uint8_t *e8m0_t;       /* [cols, rows / 32], device; tiled: see above */
  int64_t rows, cols;    /* rows % 32 == 0 */
  int32_t src_dtype;     /* GTP_F32 or GTP_BF16 */
  int32_t tiled_scales;  /* 0 or 1 (GTP_E_ARG otherwise) */
} gtp_mx_col_desc;       /* 48 bytes */

/* The columnwise views of descs[0..n) (0 <= n <= 8; a host array) in one launch, each
 * exactly as gtp_mxfp8_quantize_columnwise writes it: the views a step needs together
 * (every weight's after the optimizer step; dY's and X's before a linear's MXFP8 wgrad)
 * pay one launch's ramp and drain instead of one each.  Every descriptor is checked
 * before anything is launched (the first failure's status is returned and nothing runs).
 * A matrix whose rows do not all start on 16 bytes (cols not a multiple of 4 for F32, 8
 * for BF16, or src not 16-byte aligned) is quantized by a launch of its own before the
 * group.  No output may overlap a source or another output (GTP_E_ARG, found before
 * anything is launched); sources may be shared. */
gtp_status gtp_mxfp8_quantize_columnwise_group(const gtp_mx_col_desc *descs, int32_t n,
                                               gtp_stream stream);

/* Y[M,N] (bf16) = dq(Xq[M,K], Xs[M,K/32]) · dq(Wq[N,K], Ws[N,K/32])^T on the
 * block-scaled FP8 tensor-core path, fp32 accumulation, RNE to bf16.  Both operands
 * are quantized along K, as gtp_mxfp8_quantize_rowwise writes them.
 * K % 128 == 0 (else GTP_E_SHAPE); N % 8 == 0, so that Y's rows are 16-byte multiples
 * (else GTP_E_ALIGN); any M.  All device pointers:
 * Xq, Wq and Y 16-byte aligned, Xs and Ws 4-byte aligned (GTP_E_ALIGN otherwise) - so a
 * weight's view inside a native MXFP8 buffer (gtp_adam_step_flat_mxfp8) qualifies
 * whenever its buffer offset is a multiple of 128 elements.  Speed, not results: with
 * M > 128 the CTA-pair kernel runs; it fetches scale rows by tensor copy when K % 512 == 0
 * and both scale arrays are 16-byte aligned (a buffer offset that is a multiple of 512
 * elements), else gathers them with loads (about 10 % slower).  The same holds for the
 * dgrad and wgrad entry points below (their contraction is N and M). */
gtp_status gtp_linear_fprop_mxfp8(const uint8_t *Xq, const uint8_t *Xs, const uint8_t *Wq,
                                  const uint8_t *Ws, void *Y, int64_t M, int64_t N, int64_t K,
                                  gtp_stream stream);

/* MXFP8 dgrad ([LIN] §4.2 on the MXFP8 weight's columnwise view):
 * dX[M,K] (bf16) = dq(dYq[M,N], dYs[M,N/32]) · dq(Wtq[K,N], Wts[K,N/32])^T, with dY
 * quantized rowwise and W columnwise (gtp_mxfp8_quantize_columnwise of W[N,K]).
 * N % 128 == 0, K % 8 == 0.  All device pointers; codes and dX 16-byte aligned, scales
 * 4-byte aligned. */
gtp_status gtp_linear_dgrad_mxfp8(const uint8_t *dYq, const uint8_t *dYs, const uint8_t *Wtq,
                                  const uint8_t *Wts, void *dX, int64_t M, int64_t N, int64_t K,
                                  gtp_stream stream);

/* MXFP8 wgrad accumulated into the fp32 main_grad view ([LIN] §4.2, [BUF] §5):
 * grad_data[grad_offset : +N*K].view(N,K) += dq(dYtq[N,M], dYts[N,M/32])
 *                                            · dq(Xtq[K,M], Xts[K,M/32])^T,
 * both operands quantized along the token dimension M (the columnwise view of dY[M,N]
 * and of X[M,K]).  M % 128 == 0, K % 4 == 0, grad_offset % 4 == 0, the view inside the
 * buffer (GTP_E_RANGE).  All device pointers; codes and grad_data 16-byte aligned,
 * scales 4-byte aligned. */
gtp_status gtp_linear_wgrad_accum_mxfp8(const uint8_t *dYtq, const uint8_t *dYts,
                                        const uint8_t *Xtq, const uint8_t *Xts, float *grad_data,
                                        int64_t grad_offset, int64_t grad_numel_total, int64_t M,
                                        int64_t N, int64_t K, gtp_stream stream);

/* ----------------------------------------------------------------------- NVFP4
 * Native NVFP4 weights ([GTP] §1.3 and "GTP + NVFP4"): packed 4-bit E2M1 elements
 * (kFloat4E2M1), one E4M3 scale byte per block of 16 consecutive elements of a row
 * ("Block 16", 0.5 + 1/16 B/elem), and a per-tensor scale set when the optimizer step
 * quantizes.  The scale rule (the pages give none; NVIDIA's two-level NVFP4 recipe, every
 * step in fp32), with amax = max |x| over the tensor's finite elements:
 *   S    = 1 if amax == 0, else min(2688 / amax, FLT_MAX)          2688 = 448 * 6
 *   sf_b = RNE_E4M3_satfinite((amax_b / 6) * S)        amax_b = max |x| over the block
 *   code = RNE_E2M1_satfinite(x * min(S / sf_b, FLT_MAX)), x * 0 when sf_b == 0
 * and x ~= e2m1(code) * sf_b / S.  A block holding NaN or Inf gets scale byte 0x7F and
 * codes 0.  Two codes share a byte, the even element in the low nibble.
 */

/* src[rows,cols] (F32 or BF16) -> packed[rows, cols/2], scales[rows, cols/16] and
 * *amax (device fp32, written: the tensor amax, from which S follows).  cols % 16 == 0
 * (else GTP_E_SHAPE).  All device pointers; src and packed 16-byte aligned, amax 4-byte
 * aligned.  Two kernels plus a 4-byte memset of *amax, on `stream`. */
gtp_status gtp_nvfp4_quantize_rowwise(const void *src, gtp_dtype src_dt, int64_t rows,
                                      int64_t cols, uint8_t *packed, uint8_t *scales,
                                      float *amax, gtp_stream stream);

/* Y[M,N] (bf16) = dq(Xq[M,K/2], Xs[M,K/16], *x_amax) · dq(Wq[N,K/2], Ws[N,K/16], *w_amax)^T
 * on the block-scaled FP4 tensor-core path (kind::mxf4nvf4, E4M3 block scales), fp32
 * accumulation, times 1 / (S_x S_w), RNE to bf16.  Both operands quantized along K by
 * gtp_nvfp4_quantize_rowwise.  K % 256 == 0 (GTP_E_SHAPE), N % 8 == 0 (GTP_E_ALIGN).
 * All device pointers: Xq, Xs, Wq, Ws, Y 16-byte aligned; x_amax, w_amax 4-byte aligned. */
gtp_status gtp_linear_fprop_nvfp4(const uint8_t *Xq, const uint8_t *Xs, const float *x_amax,
                                  const uint8_t *Wq, const uint8_t *Ws, const float *w_amax,
                                  void *Y, int64_t M, int64_t N, int64_t K, gtp_stream stream);

/* ------------------------------------------------------------------ tiled scale layout
 * The block-scale arrays above are [rows, cols] bytes (cols = K/32 for MXFP8, K/16 for
 * NVFP4): one row of scales per row of codes.  The tiled layout holds the same bytes in the
 * order the block-scaled GEMMs read them, so that a pipeline stage's scales of 128 rows are
 * one contiguous copy instead of one 16-byte request per row.  The bytes of a row group
 * into 32-bit words (word w = bytes 4w .. 4w+3, little-endian); the tiled array is a
 * sequence of 512-byte atoms, atom (t, w) for row tile t = r / 128 and word w at index
 * t * ceil(cols / 4) + w; inside an atom, the word of row 128 t + 32 c + l sits at byte
 * 16 l + 4 c.  That is the order in which tcgen05.cp.32x128b.warpx4 moves a 32-row x 16-byte
 * block into the tensor-memory columns that the scale operand of a block-scaled
 * tcgen05.mma reads (word of row 32 c + l in lane l, column c).  The pages give the scales'
 * values, not their order in memory; this order is the tensor core's.
 *
 * gtp_sf_tiled_bytes: bytes of the tiled form of a [rows, cols] array,
 * ceil(rows / 128) * ceil(cols / 4) * 512; -1 if a size is negative.  Host only. */
int64_t gtp_sf_tiled_bytes(int64_t rows, int64_t cols);

/* Writes the tiled form of sf[rows, cols] (device, row-major, any alignment) into `tiled`
 * (device, gtp_sf_tiled_bytes(rows, cols) bytes, 4-byte aligned, else GTP_E_ALIGN).
 * Padding bytes (rows >= rows, columns >= cols of the last atoms) are written as zero.
 * One kernel on `stream`; nothing for an empty array. */
gtp_status gtp_sf_tile(const uint8_t *sf, int64_t rows, int64_t cols, uint8_t *tiled,
                       gtp_stream stream);

/* As gtp_mxfp8_quantize_rowwise, with the scales written in the tiled layout:
 * e8m0_tiled holds gtp_sf_tiled_bytes(rows, cols / 32) bytes (any alignment); padding
 * bytes are not written.  Codes and scale values are identical. */
gtp_status gtp_mxfp8_quantize_rowwise_tiled(const void *src, gtp_dtype src_dt, int64_t rows,
                                            int64_t cols, uint8_t *e4m3, uint8_t *e8m0_tiled,
                                            gtp_stream stream);

/* One matrix of gtp_mxfp8_quantize_rowwise_group: the arguments of
 * gtp_mxfp8_quantize_rowwise (tiled_scales 0) or gtp_mxfp8_quantize_rowwise_tiled
 * (tiled_scales 1), with the same meaning and rules. */
typedef struct {
  const void *src;       /* [rows, cols] F32 or BF16, device, 16-byte aligned */
  uint8_t *e4m3;         /* [rows, cols], device, 16-byte aligned */
  uint8_t *e8m0;         /* [rows, cols / 32], or the tiled layout */
  int64_t rows, cols;    /* cols % 32 == 0 */
  int32_t src_dtype;     /* GTP_F32 or GTP_BF16 */
  int32_t tiled_scales;  /* 0 or 1 (GTP_E_ARG otherwise) */
} gtp_mx_row_desc;       /* 48 bytes */

/* The rowwise quantizations of descs[0..n) (0 <= n <= 8; a host array) in one launch, each
 * exactly as its single call writes it: the matrices a step quantizes together (the
 * updated masters after the optimizer step, a layer's inputs) pay one launch's ramp and
 * drain.  Every descriptor is checked before anything is launched; no output may overlap
 * a source or another output (GTP_E_ARG); sources may be shared. */
gtp_status gtp_mxfp8_quantize_rowwise_group(const gtp_mx_row_desc *descs, int32_t n,
                                            gtp_stream stream);

/* As gtp_nvfp4_quantize_rowwise, with the scales written in the tiled layout:
 * scales_tiled holds gtp_sf_tiled_bytes(rows, cols / 16) bytes (any alignment); padding
 * bytes are not written.  Codes, scale values and the amax are identical. */
gtp_status gtp_nvfp4_quantize_rowwise_tiled(const void *src, gtp_dtype src_dt, int64_t rows,
                                            int64_t cols, uint8_t *packed, uint8_t *scales_tiled,
                                            float *amax, gtp_stream stream);

/* As gtp_linear_fprop_mxfp8 and gtp_linear_fprop_nvfp4, with both scale arrays in the
 * tiled layout (Xs_tiled: rows M, Ws_tiled: rows N; 16-byte aligned, else GTP_E_ALIGN).
 * The same products bit for bit.  Always the CTA-pair kernel: its producer copies each
 * stage's scale atoms with the operands (three tensor copies a stage), and no warp
 * rearranges scale bytes. */
gtp_status gtp_linear_fprop_mxfp8_tiled(const uint8_t *Xq, const uint8_t *Xs_tiled,
                                        const uint8_t *Wq, const uint8_t *Ws_tiled, void *Y,
                                        int64_t M, int64_t N, int64_t K, gtp_stream stream);
gtp_status gtp_linear_fprop_nvfp4_tiled(const uint8_t *Xq, const uint8_t *Xs_tiled,
                                        const float *x_amax, const uint8_t *Wq,
                                        const uint8_t *Ws_tiled, const float *w_amax, void *Y,
                                        int64_t M, int64_t N, int64_t K, gtp_stream stream);

/* As gtp_linear_dgrad_mxfp8 and gtp_linear_wgrad_accum_mxfp8, with both scale arrays in
 * the tiled layout (16-byte aligned, else GTP_E_ALIGN): dgrad takes dYs_tiled (rows M,
 * from gtp_mxfp8_quantize_rowwise_tiled of dY) and Wts_tiled (rows K, from
 * gtp_mxfp8_quantize_columnwise_tiled of W); wgrad takes dYts_tiled (rows N) and Xts_tiled
 * (rows K), both from gtp_mxfp8_quantize_columnwise_tiled.  The same products bit for bit
 * as the [rows, cols]-scale entry points on the CTA-pair kernel (the tiled forms always
 * run it); wgrad accumulates in fp32 as gtp_linear_wgrad_accum_mxfp8 does, with the same
 * argument rules. */
gtp_status gtp_linear_dgrad_mxfp8_tiled(const uint8_t *dYq, const uint8_t *dYs_tiled,
                                        const uint8_t *Wtq, const uint8_t *Wts_tiled, void *dX,
                                        int64_t M, int64_t N, int64_t K, gtp_stream stream);
gtp_status gtp_linear_wgrad_accum_mxfp8_tiled(const uint8_t *dYtq, const uint8_t *dYts_tiled,
                                              const uint8_t *Xtq, const uint8_t *Xts_tiled,
                                              float *grad_data, int64_t grad_offset,
                                              int64_t grad_numel_total, int64_t M, int64_t N,
                                              int64_t K, gtp_stream stream);

/* ------------------------------------------- the all-to-all reduce-scatter's local sum
 * [BUF] §9.1 (reduce_scatter_with_fp32_accumulation): the bucket's reduce-scatter is an
 * all-to-all in which each rank receives the P = world_size low-precision slices of its
 * own shard; it then adds them with an fp32 sum and casts the total to the output dtype.
 * This is that sum on the receiving GPU:
 *   out[i] = cast_out(slice_0[i] + slice_1[i] + ... + slice_{P-1}[i]),
 * accumulated in fp32 in rank order, one fp32 rounding per addition (deterministic), and
 * rounded once to nearest even for a bf16 output.
 * slices: host array of P (1 to 128) device pointers to n elements each, of in_dt
 * (GTP_BF16 or GTP_F32), 16-byte aligned; out: n elements of out_dt (GTP_BF16 or GTP_F32),
 * device, 16-byte aligned.  out may be one of the slices exactly (same start, same dtype),
 * but may not overlap one partly (GTP_E_ARG).  One kernel on `stream`; nothing for n == 0. */
gtp_status gtp_rs_local_sum(const void *const *slices, int32_t P, int64_t n, gtp_dtype in_dt,
                            void *out, gtp_dtype out_dt, gtp_stream stream);

/* The same for an all-to-all receive buffer held as one array: slice r starts at
 * slices + r * row_bytes (row_bytes a multiple of 16 with a 16-byte aligned base, else
 * GTP_E_ALIGN; the slices may not overlap: row_bytes >= n x the element size when P > 1,
 * else GTP_E_ARG).  Arguments otherwise as gtp_rs_local_sum. */
gtp_status gtp_rs_local_sum_rows(const void *slices, int64_t row_bytes, int32_t P, int64_t n,
                                 gtp_dtype in_dt, void *out, gtp_dtype out_dt, gtp_stream stream);

/* ------------------------------------------------------------------ diagnostics
 * Every wait inside the tensor-core kernels has a time limit.  A wait that runs out sets
 * a bit in a per-device word and the kernel unwinds (its results are then invalid):
 * bit 0 operand ring (producer side), bit 1 accumulator hand-off, bit 2 operand ring
 * (MMA side), bit 3 epilogue, bit 5/6 the dynamic schedule's ring, bit 7 a drain of the
 * kernel's own copies at exit, bit 8 the self-test below.
 * Reads the word into *flags (host pointer) and clears it if reset != 0.  Synchronous
 * with respect to the current device.  The pages' failure detection ("05 · grad/param
 * buffer ...", §6.3: NaN / large-gradient checks before the collective) is a check of the
 * gradients; this word is the device-side half of the same idea for the kernels' own
 * waits, which the pages do not describe. */
gtp_status gtp_wait_timeouts(uint32_t *flags, int32_t reset);

/* Self-test of the bounded waits: launches one 32-thread block on `stream` in which one
 * thread waits, through the same bounded wait the tensor-core kernels use, on an mbarrier
 * that nothing arrives on, with a limit of limit_ns nanoseconds (1e3 .. 1e8, else
 * GTP_E_ARG).  The wait runs out, sets bit 8 of the word gtp_wait_timeouts reads, and the
 * kernel returns normally: nothing faults, traps or hangs, and the context stays usable.
 * Asynchronous; the bit is visible once the stream has reached the kernel.  Tests use it
 * to show that an expired wait is reported and survived. */
gtp_status gtp_selftest_wait_timeout(int64_t limit_ns, gtp_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* GTP_H_ */
