/*
 * zero.h -- C ABI of libzero.so, the GB300 (sm_103a) ZeRO-DP optimizer step.
 *
 * One GPU simulates n_d data-parallel ranks: each rank is a gradient buffer
 * in HBM.  A step reduce-scatters the ranks' 16-bit gradients (rank-ordered
 * fp32 sum divided by n_d times the loss scale), applies mixed-precision Adam
 * to each shard's fp32 master weights, momentum and variance, and all-gathers
 * the updated weights as 16-bit values.
 *
 * Sources (page title, section):
 *   DP-notes  "Data parallelism and ZeRO optimization -- Hinglish notes" (6.1.8)
 *   LLM-par   "大模型并行技术" (LLM parallelism techniques)
 *   itwiki    "ZeRO (딥 러닝)"
 *
 * Conventions for every call below.
 *   - Pointers named *_dev / device buffers are device pointers of the current
 *     device; the caller allocates and owns all of them.  No call allocates
 *     device memory and no call synchronises the stream.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Every kernel is launched on it; results are ready when it is.
 *   - Device pointers must be 16-byte aligned (ZERO_ERR_MISALIGNED otherwise);
 *     the workspace and the scalars block 256-byte aligned.
 *   - Argument errors are returned synchronously and launch nothing.  A failed
 *     launch returns ZERO_ERR_CUDA.  Errors found on the device (a bounded wait
 *     that ran out) are OR-ed into zero_dev_scalars.status as ZERO_DEV_*.
 *   - Index domain: Psi parameters, split into n_d contiguous shards of S
 *     elements, S = roundup(ceil(Psi / n_d), shard_pad); shard r covers global
 *     [r*S, min((r+1)*S, Psi)).  Arrays "of n_d*S" are indexed by the global
 *     index j for j < Psi; their entries in [Psi, n_d*S) are padding that no
 *     call changes (zero them once; they stay zero).  Rank gradient buffers
 *     hold at least Psi elements; nothing past Psi is read.  A gathered buffer
 *     is written only in [0, Psi).
 *   - A plan is host memory only, immutable after creation, safe to share
 *     between threads.  Calls that share a workspace or a scalars block must
 *     be ordered on one stream.
 */
#ifndef ZERO_H
#define ZERO_H

#include <stddef.h>

#if defined(__GNUC__)
#define ZERO_API __attribute__((visibility("default")))
#else
#define ZERO_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define ZERO_ABI_VERSION 2
#define ZERO_MAX_RANKS 256      /* largest n_d */
#define ZERO_MAX_SHARD_PAD 4096 /* largest shard_pad */
#define ZERO_MAX_MICRO_BATCHES 65536 /* largest gradient-accumulation count */
#define ZERO_MAX_LAYERS 65536   /* largest layer count of zero_step_layers */

typedef enum {
    ZERO_OK = 0,
    ZERO_ERR_INVALID_ARG = 1, /* a size, a dtype, a stage or a NULL pointer is wrong  */
    ZERO_ERR_MISALIGNED = 2,  /* a device pointer breaks the alignment rule above     */
    ZERO_ERR_UNSUPPORTED = 3, /* a valid request the library does not implement       */
    ZERO_ERR_CUDA = 4,        /* the CUDA runtime reported an error at launch         */
    ZERO_ERR_TIMEOUT = 5,     /* a bounded device wait ran out (see ZERO_DEV_TIMEOUT) */
    ZERO_ERR_BOUNDS = 6       /* a request exceeds a fixed capacity of the library   */
} zero_status;

typedef enum { ZERO_BF16 = 0, ZERO_FP16 = 1 } zero_dtype;

/* bits of zero_dev_scalars.status */
#define ZERO_DEV_TIMEOUT 1 /* a bounded wait inside a kernel ran out; that kernel stopped early */

typedef struct zero_plan zero_plan;

/* Optional plan settings (zero_plan_create_ex).  Zero-initialised = defaults. */
typedef struct {
    int param_dtype_set;           /* 0: parameters are bf16; 1: use param_dtype              */
    zero_dtype param_dtype;        /* dtype of the gathered / sharded 16-bit parameters       */
    long long reduce_bucket_elems; /* itwiki DeepSpeed config "reduce_bucket_size": the fused
                                      step runs in buckets of at most this many parameters;
                                      <= 0 means one bucket.  Rounded up to 2048.            */
} zero_plan_opts;

/* Adam hyper-parameters, copied by value at each call.  Adam itself is not
 * printed on the pages (DP-notes "Memory Consumption Analysis" sizes its fp32
 * momentum, variance and master copy); the update is textbook Adam (bias
 * correction, eps outside the square root) in the efficient order Kingma &
 * Ba give for their Algorithm 1, with decoupled weight decay (AdamW) when
 * weight_decay > 0.  With s = sqrt(1-b2^t):
 *     p <- p * (1 - lr*wd)              (only when wd != 0)
 *     m <- b1*m + (1-b1)*g
 *     v <- b2*v + (1-b2)*(g*g)
 *     p <- p - ((lr*s)/(1-b1^t)) * (m / (sqrt(v) + eps*s))
 * each operation one IEEE fp32 rounding, in this order (equal to Algorithm 1
 * in exact arithmetic).                                                      */
typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
    float max_norm;   /* > 0: clip the averaged gradient to this global L2 norm
                         (itwiki DeepSpeed config "gradient_clipping"); coef =
                         max_norm/(norm+1e-6), applied when < 1                   */
    int loss_scaling; /* 1: fp16 dynamic loss scaling: the divisor includes the
                         loss scale; a step with a non-finite averaged gradient is
                         skipped, the scale halves (floor min_scale); after
                         scale_window good steps in a row it doubles              */
    int scale_window; /* e.g. 1000 */
    float min_scale;  /* e.g. 1 */
} zero_hparams;

/* Step scalars, resident in device memory (64 bytes, 256-byte aligned),
 * written by zero_scalars_init and advanced by every step call.             */
typedef struct {
    long long t;          /* committed steps (skipped steps do not count)          */
    double beta1_pow;     /* beta1^t as a running fp64 product                     */
    double beta2_pow;     /* beta2^t                                               */
    double sqnorm;        /* squared L2 norm of the averaged gradient (clipping)   */
    float loss_scale;     /* current loss scale                                    */
    float clip_coef;      /* coefficient applied in the latest step, 1 if none     */
    int good_steps;       /* consecutive committed steps since the scale changed   */
    int overflow;         /* 1 if the latest step was skipped                      */
    int status;           /* sticky ZERO_DEV_* bits                                */
    int nonfinite;        /* internal: the step in flight saw a non-finite value   */
    unsigned int ctas_done; /* internal: CTAs of the kernel in flight that finished;
                               0 between calls                                     */
    int reserved;
} zero_dev_scalars;

/* ---------------------------------------------------------------- misc --- */
ZERO_API const char* zero_status_str(zero_status s);
ZERO_API int zero_abi_version(void);
ZERO_API size_t zero_dev_scalars_size(void);

/* ---------------------------------------------------------------- plan --- */
/* Partition of Psi parameters over n_d ranks (DP-notes "ZeRO-1: Optimizer
 * State Partitioning": theta = [theta_1 .. theta_N], rank r owns theta_r;
 * itwiki "FSDP와의 관계": flatten, then shard).  stage 1, 2 or 3 (itwiki
 * "ZeRO-DP의 세 단계"): stages 1-2 write the updated parameters into a
 * gathered buffer of Psi, stage 3 into a sharded buffer of n_d*S; the math
 * is the same.  1 <= n_d <= ZERO_MAX_RANKS, Psi >= 1,
 * 1 <= shard_pad <= ZERO_MAX_SHARD_PAD.  *out receives a new plan.          */
ZERO_API zero_status zero_plan_create(zero_plan** out, long long psi, int n_d, int stage,
                                      zero_dtype grad_dtype, int shard_pad);
ZERO_API zero_status zero_plan_create_ex(zero_plan** out, long long psi, int n_d, int stage,
                                         zero_dtype grad_dtype, int shard_pad,
                                         const zero_plan_opts* opts);
ZERO_API void zero_plan_destroy(zero_plan* plan);

/* shard_size = S, padded_psi = n_d*S; valid_len (host array of n_d, or NULL)
 * receives each shard's valid length min(max(Psi - r*S, 0), S).             */
ZERO_API zero_status zero_plan_query(const zero_plan* plan, long long* shard_size,
                                     long long* padded_psi, long long* valid_len);

/* Model-state bytes per rank at `stage` (0..3) with K optimizer bytes per
 * parameter (itwiki memory table: 2 + 2 + K, K = 12; stage table: stage 1
 * divides K*Psi by n_d, stage 2 also the gradients, stage 3 also the
 * parameters).  bytes_out[4] = {params, grads, optimizer, total}.            */
ZERO_API zero_status zero_plan_memory(const zero_plan* plan, int stage, double k,
                                      double bytes_out[4]);

/* Elements each rank sends per step at `stage` (itwiki "왜 통신량이 늘지
 * 않는가": reduce-scatter Psi + all-gather Psi; stage 3 gathers twice).     */
ZERO_API zero_status zero_plan_comm_volume(const zero_plan* plan, int stage, double* elems_out);

/* Bytes of workspace the calls below need with these hyper-parameters (an
 * upper bound valid on every device).  Only the step and reduce calls use it.*/
ZERO_API size_t zero_workspace_bytes(const zero_plan* plan, const zero_hparams* hp);

/* Write initial step scalars: t = 0, beta powers 1, loss_scale, counters 0.  */
ZERO_API zero_status zero_scalars_init(zero_dev_scalars* scalars_dev, float loss_scale,
                                       void* stream);

/* ------------------------------------------------------ step, in parts --- */
/* Reduce-scatter (DP-notes "ZeRO-2: Gradient Partitioning": rank r receives
 * the averaged gradient of its partition; itwiki FSDP reduces in fp32):
 *   grad_shards[j] = (sum over ranks q = 0..n_d-1, in order, from +0.0f, of
 *                     float(rank_grads[q][j])) / D,   j < Psi
 * with D = (float)n_d * (hp->loss_scaling ? loss_scale : 1).
 * rank_grads: host array of n_d device pointers (plan grad dtype, >= Psi
 * elements each).  grad_shards: n_d*S floats; its padding is set to +0.
 * Also leaves per-block partial sums of grad_shards[j]^2 in `ws` for
 * zero_grad_sqnorm, and, in loss-scaling mode, records a non-finite value in
 * scalars->nonfinite for the following Adam call.                           */
ZERO_API zero_status zero_reduce_scatter(const zero_plan* plan, const void* const* rank_grads,
                                         const zero_hparams* hp, zero_dev_scalars* scalars_dev,
                                         float* grad_shards, void* ws, void* stream);

/* Global squared L2 norm of the averaged gradient, sum over j < Psi of
 * grad_shards[j]^2, into scalars->sqnorm; with hp->max_norm > 0 also
 * scalars->clip_coef = coef when coef < 1, else 1.  grad_shards == NULL:
 * finish the partial sums the preceding zero_reduce_scatter left in ws
 * (no second read of the gradient).  Deterministic for a given device.      */
ZERO_API zero_status zero_grad_sqnorm(const zero_plan* plan, const float* grad_shards,
                                      const zero_hparams* hp, zero_dev_scalars* scalars_dev,
                                      void* ws, void* stream);

/* Adam on every shard (DP-notes "ZeRO-1": rank r updates only theta_r with
 * its local optimizer states), in place on master/m/v (n_d*S floats each),
 * from grad_shards (n_d*S).  With hp->max_norm > 0 the gradient is first
 * multiplied by scalars->clip_coef.  In loss-scaling mode a step flagged
 * non-finite by the preceding reduce is skipped.  lp_out (NULL: none): the
 * 16-bit cast of the updated master, at index j < Psi -- the gathered buffer
 * for stages 1-2, the sharded buffer (n_d*S) for stage 3.  Commits the step
 * scalars (t, beta powers, loss scale).                                      */
ZERO_API zero_status zero_adam_shard_step(const zero_plan* plan, const zero_hparams* hp,
                                          const float* grad_shards, float* master, float* m,
                                          float* v, void* lp_out, zero_dev_scalars* scalars_dev,
                                          void* stream);

/* All-gather (DP-notes "ZeRO-1": updated partitions are gathered so every
 * rank holds the full model; itwiki: ZeRO-3 gathers each layer before use):
 * gathered[r*S + i] = shards_lp[r][i] for i < valid_len(r).  shards_lp: host
 * array of n_d device pointers to S 16-bit values (plan parameter dtype),
 * each needing only 2-byte alignment (shards cut from one flat n_d*S buffer
 * at any S are accepted; the fast path wants 16-byte aligned shards).
 * scalars_dev (may be NULL) receives ZERO_DEV_TIMEOUT if a wait runs out.   */
ZERO_API zero_status zero_all_gather(const zero_plan* plan, const void* const* shards_lp,
                                     void* gathered, zero_dev_scalars* scalars_dev, void* stream);

/* --------------------------------------------------------- fused step --- */
/* The whole step in as few passes as the global checks allow: reduce-scatter,
 * Adam and the 16-bit cast written straight to lp_out (gathered buffer for
 * stages 1-2, sharded buffer for stage 3), the reduced gradient kept in
 * registers.  State is read from *_in and written to *_out (each n_d*S); the
 * *_out may equal their *_in (all three or none); otherwise no *_out may
 * share a byte with another state array (ZERO_ERR_INVALID_ARG).  Passes:
 *   no clipping, no loss scaling : 1 pass
 *   loss scaling, out != in      : 1 pass, speculative; on overflow the out
 *                                  state is restored from in and lp_out is
 *                                  re-cast from master_in
 *   loss scaling, out == in      : a read-only check pass, then the update
 *   clipping                     : a reduce pass (writes the fp32 reduced
 *                                  gradient to ws when n_d > 4, else only the
 *                                  norm), then the update
 * In every case, after the call lp_out[j] (j < Psi) is the 16-bit cast of
 * master_out[j] if the call wrote it, and scalars are advanced.  Runs in
 * buckets of the plan's reduce_bucket_elems when no global check is needed.  */
ZERO_API zero_status zero_step_fused(const zero_plan* plan, const zero_hparams* hp,
                                     const void* const* rank_grads, const float* master_in,
                                     const float* m_in, const float* v_in, float* master_out,
                                     float* m_out, float* v_out, void* lp_out,
                                     zero_dev_scalars* scalars_dev, void* ws, void* stream);

/* ZeRO-Offload on a Grace-Blackwell node (itwiki "후속 기법", ZeRO-Offload
 * row: the optimizer state moves to CPU memory).  The same step as
 * zero_step_fused, with master/m/v (in and out) in page-locked host memory
 * that the kernels read and write directly over the CPU-GPU link instead of
 * HBM; gradients, the 16-bit parameters and the workspace stay in device
 * memory.  The update still runs on the GPU.  Every state pointer must be
 * page-locked host memory mapped at the same address on the device
 * (cudaHostAlloc / torch pin_memory); anything else is refused with
 * ZERO_ERR_INVALID_ARG before a launch.  Saves 12 bytes of HBM per
 * parameter; the state's 24 bytes per parameter cross the CPU-GPU link.    */
ZERO_API zero_status zero_step_fused_offload(const zero_plan* plan, const zero_hparams* hp,
                                             const void* const* rank_grads, const float* master_in,
                                             const float* m_in, const float* v_in, float* master_out,
                                             float* m_out, float* v_out, void* lp_out,
                                             zero_dev_scalars* scalars_dev, void* ws, void* stream);

/* ------------------------------------------------ gradient accumulation --- */
/* Gradient accumulation over k micro-batches per optimizer step (DP-notes
 * "Connections": accumulation combined with ZeRO for larger effective
 * batches; itwiki "DeepSpeed에서 쓰기": gradient_accumulation_steps).  Each
 * micro-batch is reduce-scattered as it arrives, and its fp32 rank sum is
 * added to the owners' fp32 accumulator, so no rank keeps more than its
 * micro-batch gradients; the step at the k-th micro-batch divides once.     */

/* One micro-batch (not the last): acc_out[j] = acc_in[j] + sum_r g_r[j] for
 * j < Psi, the rank sum in fp32 in rank order from +0.0f, NOT divided.
 * acc_in NULL means +0.0f (the first micro-batch); acc_in may equal acc_out,
 * any other overlap is refused (ZERO_ERR_INVALID_ARG).  Both are fp32 device
 * buffers of at least Psi elements (n_d*S recommended, so that shard r of
 * the accumulator is [r*S, (r+1)*S)), 16-byte aligned; elements from Psi on
 * are not touched.  rank_grads as in zero_reduce_scatter.  One kernel.
 * scalars_dev (may be NULL) only receives ZERO_DEV_TIMEOUT if a wait runs
 * out; nothing else of it is read or written.                              */
ZERO_API zero_status zero_accumulate_grads(const zero_plan* plan, const void* const* rank_grads,
                                           const float* acc_in, float* acc_out,
                                           zero_dev_scalars* scalars_dev, void* stream);

/* The step at the last (k-th, micro_batches = k) micro-batch: rank_grads are
 * that micro-batch's gradients, acc the sum zero_accumulate_grads left for
 * micro-batches 1..k-1 (NULL exactly when k == 1).  The reduced gradient is
 * (acc[j] + sum_r g_r[j]) / (n_d * k * loss_scale) -- the mean over all
 * n_d * k rank gradients -- and everything else (clipping, loss-scale skip,
 * pass schedules, outputs) is zero_step_fused.  acc is read, never written,
 * and must not overlap an output.  1 <= k <= ZERO_MAX_MICRO_BATCHES.        */
ZERO_API zero_status zero_step_fused_accum(const zero_plan* plan, const zero_hparams* hp,
                                           const void* const* rank_grads, const float* acc, int micro_batches,
                                           const float* master_in, const float* m_in, const float* v_in,
                                           float* master_out, float* m_out, float* v_out, void* lp_out,
                                           zero_dev_scalars* scalars_dev, void* ws, void* stream);

/* ----------------------------------------------------- quantized gather --- */
/* ZeRO++ qwZ (itwiki "후속 기법", ZeRO++ row: weights are block-quantized for
 * the all-gather).  Per block of `block` consecutive elements of a shard
 * (blocks start at each shard's first element; a shard's last block may be
 * short): amax = max |x|, s = amax/127, code = clamp(rint(x/s), -127, 127)
 * (0 when s = 0), dequantized = bf16(code * s).  shards_bf16: n_d*S bf16
 * (flat).  codes_out: n_d*S int8, written for j < Psi.  scales_out:
 * n_d*ceil(S/block) floats, shard-major, 0 for blocks past a shard's valid
 * length.  gathered_bf16: Psi bf16 dequantized values (the owner's shard
 * too).  32 <= block <= 65536, block a multiple of 32.                       */
ZERO_API zero_status zero_quant_gather(const zero_plan* plan, const void* shards_bf16, int block,
                                       signed char* codes_out, float* scales_out,
                                       void* gathered_bf16, void* stream);

/* The fused step of zero_step_fused whose epilogue is the quantized gather
 * above instead of the plain 16-bit write: codes, scales and dequantized bf16
 * gathered values come from the updated master of each block (block must be
 * 2048; parameter dtype bf16).  With clipping or loss scaling a reduce pass
 * comes first (squared-norm partials and the non-finite flag, in ws:
 * zero_workspace_bytes(plan, hp) bytes, 256-byte aligned; with clipping and
 * n_d > 4 also the fp32 reduced gradient); the update pass then reads that
 * reduced gradient (or, without it, re-reads the rank gradients), finishes
 * the norm in its prologue, and with the flag set writes nothing (state,
 * codes, scales and gathered values keep the last step's) while the scalar
 * epilogue halves the scale.
 * Loss scaling needs the state in place (master_out == master_in, likewise
 * m, v), else ZERO_ERR_UNSUPPORTED.  ws may be NULL with neither.           */
ZERO_API zero_status zero_step_fused_qgather(const zero_plan* plan, const zero_hparams* hp,
                                             const void* const* rank_grads,
                                             const float* master_in, const float* m_in,
                                             const float* v_in, float* master_out, float* m_out,
                                             float* v_out, int block, signed char* codes_out,
                                             float* scales_out, void* gathered_bf16,
                                             zero_dev_scalars* scalars_dev, void* ws,
                                             void* stream);

/* ------------------------------------------- quantized gradient exchange --- */
/* ZeRO++ qgZ (itwiki "후속 기법", ZeRO++ row: gradients are quantized and
 * averaged through an all-to-all; bit width and blocking not given).  The
 * reading: every rank quantizes its own gradient with the block quantizer of
 * zero_quant_gather (int8, absmax/127 scale, blocks aligned to each
 * destination shard's start), only codes and scales travel, and the shard
 * owner reconstructs each rank's value as (float)code * scale (one fp32
 * rounding) before the rank-ordered fp32 sum.
 *
 * Sender side: rank q's bf16 gradient (>= Psi elements) -> int8 codes at the
 * global index j < Psi and fp32 block scales.  rank_codes: host array of n_d
 * device pointers (>= Psi int8 each, 16-byte aligned).  rank_scales: one
 * array of n_d * ceil(S/block) rows of n_dp = roundup(n_d, 4) floats, block-
 * major and rank-minor: rank q's scale of block b of shard r at
 * [(r * ceil(S/block) + b) * n_dp + q] (so one tile's scales of all ranks
 * are contiguous); 0 for blocks past a shard's valid length and for the
 * padding columns q >= n_d.  Plan gradient dtype bf16; 32 <= block <= 65536,
 * a multiple of 32.  One kernel for all ranks; with block 2048 and a shard
 * size that is a multiple of 8, full blocks are staged by 1-D bulk copies.
 * scalars_dev (may be NULL, else 256-byte aligned) only receives
 * ZERO_DEV_TIMEOUT if a bounded wait runs out; nothing else of it is read or
 * written.                                                                  */
ZERO_API zero_status zero_quantize_grads(const zero_plan* plan, const void* const* rank_grads, int block,
                                         signed char* const* rank_codes, float* rank_scales,
                                         zero_dev_scalars* scalars_dev, void* stream);

/* Receiver side, fused: zero_step_fused with the ranks' int8 codes and
 * scales (layout as above, block 2048) in place of their 16-bit gradients:
 *   g[j] = (sum over q in order, from +0.0f, of (float)code_q[j] * scale_q(j)) / n_d
 * then Adam, cast and gather as in zero_step_fused.  With clipping
 * (hp->max_norm > 0) the schedule is zero_step_fused's: a reduce pass over the
 * codes writes the squared-norm partials (and, for n_d > 4, the reduced
 * gradient) into ws, and the update pass finishes the norm in its prologue.
 * ws: zero_workspace_bytes(plan, hp) bytes, 256-byte aligned, required with
 * clipping, unused (may be NULL) without.  Loss scaling is refused
 * (ZERO_ERR_UNSUPPORTED): the sender takes bf16 gradients, which need none. */
ZERO_API zero_status zero_step_fused_qgz(const zero_plan* plan, const zero_hparams* hp,
                                         const signed char* const* rank_codes, const float* rank_scales,
                                         int block, const float* master_in, const float* m_in,
                                         const float* v_in, float* master_out, float* m_out, float* v_out,
                                         void* lp_out, zero_dev_scalars* scalars_dev, void* ws,
                                         void* stream);

/* The ZeRO++ step with both quantized collectives: the receiver of
 * zero_step_fused_qgz (the ranks' int8 codes and scales in, dequantized and
 * summed in rank order, Adam) whose epilogue is the quantized gather of
 * zero_step_fused_qgather (codes_out, scales_out and the dequantized bf16
 * gathered values from the updated master, blocks of 2048 from each shard's
 * first element).  Layouts as in those two entry points.  With clipping a
 * reduce pass over the codes comes first (norm partials in ws:
 * zero_workspace_bytes(plan, hp) bytes, 256-byte aligned; ws may be NULL
 * without clipping); for n_d > 4 it also writes the fp32 reduced gradient,
 * which the update pass reads, else the update pass re-reads the codes.  block must be 2048,
 * the parameter dtype bf16; no loss scaling (ZERO_ERR_UNSUPPORTED).         */
ZERO_API zero_status zero_step_fused_qgz_qgather(const zero_plan* plan, const zero_hparams* hp,
                                                 const signed char* const* rank_codes, const float* rank_scales,
                                                 int block, const float* master_in, const float* m_in,
                                                 const float* v_in, float* master_out, float* m_out,
                                                 float* v_out, signed char* codes_out, float* scales_out,
                                                 void* gathered_bf16, zero_dev_scalars* scalars_dev, void* ws,
                                                 void* stream);

/* ------------------------------------------------------- ZeRO-3 layer loop --- */
/* One ZeRO-3 step over a stack of layers (itwiki "ZeRO-DP의 세 단계" and
 * "왜 통신량이 늘지 않는가": with stage 3 each layer's parameters are
 * all-gathered before they are used, in the forward and again in the
 * backward pass, and each layer's gradients are reduce-scattered to their
 * owners; itwiki "DeepSpeed에서 쓰기": its example configuration is stage 3
 * with gradient_clipping 1.0, gradient_accumulation_steps, overlap_comm and
 * the stage-3 prefetch, which overlaps the next layer's gather with the
 * current layer's work).
 *
 * Per layer l = 0 .. n_layers-1, in order:
 *   gather(l): zero_all_gather of layer l's 16-bit shards into
 *              gathered[l % n_gathered], `gathers` times (1: once per step;
 *              2: forward and backward, the pages' 3-Psi volume); with
 *              gathered_codes and gathered_scales (itwiki "후속 기법",
 *              ZeRO++ row: qwZ block-quantizes the weight all-gather) it is
 *              zero_quant_gather with block 2048 instead: codes into
 *              gathered_codes[k] (n_d*S_l int8), scales into
 *              gathered_scales[k] (n_d*ceil(S_l/2048) floats), dequantized
 *              bf16 into gathered[k], k = l % n_gathered (bf16 parameters);
 *   step(l):   zero_step_fused_accum of layer l in place (stage 3: the
 *              updated 16-bit shards overwrite shards_lp).
 * gather(l) reads the shards as the previous step left them; step(l) comes
 * after gather(l).  With gather_stream a stream other than `stream` (and
 * n_gathered >= 2), every gather runs on gather_stream, ordered by events:
 * gather(l+1) is issued before step(l) so the two overlap, gather(l) waits
 * for step(l - n_gathered) (the last user of its buffer), step(l) waits for
 * gather(l), and `stream` waits for gather_stream at the end; the call's work
 * is complete when `stream` is.  gather_stream NULL (or n_gathered 1): all
 * on `stream`, gather(l+1) after step(l).  The results do not depend on the
 * schedule.
 *
 * The stack is one model: its step scalars (one block) are committed once
 * per call, so every layer's Adam takes the same t, and the global checks
 * span every layer.  With clipping the norm is that of the whole stack's
 * averaged gradient, the same coefficient for every layer; with loss scaling
 * a non-finite value in any layer skips the step for all of them (and the
 * scale halves).  Then a reduce pass over every layer comes first (norm
 * partials, the non-finite flag, and with clipping and n_d > 4 the fp32
 * reduced gradient, which the update pass reads instead of the ranks), the
 * norm is finished once, and the updates follow.  ws: with clipping or loss
 * scaling, zero_layers_workspace_bytes(hp, n_layers, layers) bytes, 256-byte
 * aligned (NULL allowed without either).
 *
 * micro_batches = k (gradient accumulation, as zero_step_fused_accum): each
 * layer's rank_grads are its k-th micro-batch's gradients, acc the sum
 * zero_accumulate_grads left for micro-batches 1..k-1 (NULL exactly when
 * k == 1); the mean divides by n_d * k.
 *
 * Each layer has its own stage-3 plan; all plans share n_d and the dtypes.
 * gathered: host array of n_gathered device pointers (1 <= n_gathered <=
 * n_layers), buffer k holding at least Psi_l 16-bit values for every layer l
 * with l % n_gathered == k.  Per layer: rank_grads as in zero_step_fused;
 * master, m, v of n_d*S_l floats, updated in place; shards_lp n_d*S_l 16-bit
 * (plan parameter dtype), 16-byte aligned.  A layer with state_on_host
 * keeps master/m/v in page-locked host memory mapped at the same address
 * (else ZERO_ERR_INVALID_ARG).  Events are created and released inside the
 * call; no device memory is allocated.                                     */
typedef struct {
    const zero_plan* plan;         /* this layer's partition, stage 3             */
    const void* const* rank_grads; /* host array of n_d device pointers           */
    const float* acc;              /* accumulated earlier micro-batches, or NULL  */
    float* master;                 /* n_d*S fp32, in place                        */
    float* m;
    float* v;
    void* shards_lp;               /* n_d*S 16-bit parameter shards, flat         */
    void* grads_ready;             /* cudaEvent_t or NULL: the layer's first read
                                      of its gradients waits for it (the copy or
                                      backward pass that wrote them)              */
    void* stepped;                 /* cudaEvent_t or NULL: recorded on `stream`
                                      after step(l) (its gradient buffers may be
                                      refilled, its shards read, from then on)    */
    int state_on_host;             /* 1: master, m, v are page-locked host memory
                                      read and written over the CPU-GPU link, as
                                      in zero_step_fused_offload (itwiki DeepSpeed
                                      example: offload_optimizer to the CPU)     */
} zero_layer;

/* Workspace bytes zero_step_layers needs with these hyper-parameters and
 * layers (the same on every device); 0 for invalid arguments.               */
ZERO_API size_t zero_layers_workspace_bytes(const zero_hparams* hp, int n_layers, const zero_layer* layers);

ZERO_API zero_status zero_step_layers(const zero_hparams* hp, int n_layers, const zero_layer* layers,
                                      int micro_batches, int gathers, int n_gathered, void* const* gathered,
                                      signed char* const* gathered_codes, float* const* gathered_scales,
                                      zero_dev_scalars* scalars_dev, void* ws, void* stream, void* gather_stream);

/* ----------------------------------------------------------- diagnostics --- */
/* Launch one kernel that waits on a barrier nothing completes, with a wait
 * limit of timeout_ns (at most 10 s).  When the limit runs out the kernel sets
 * ZERO_DEV_TIMEOUT in scalars->status and returns, leaving the context usable.
 * Exists so that the bounded-wait path can be tested.                       */
/* A pipelined kernel's own timeout path: one small launch of
 *   kernel 0: the streaming engine (reduce op, one 4096-element tile),
 *   kernel 1: the all-gather ring (one 8192-element shard),
 *   kernel 2: the gradient sender (one 2048-element block),
 *   kernel 3: the quantized weight gather (one 2048-element shard),
 * whose bulk copies are never issued, so every bounded wait runs out (after
 * timeout_ns for kernel 0, at most 10 s; after 2 ms for kernels 1 to 3).
 * Kernels 0 to 2 give up, let nothing in flight land (nothing was issued),
 * set ZERO_DEV_TIMEOUT in scalars->status and return.  scratch: a 16-byte
 * aligned device buffer of at least 32 KB; for kernels 0 to 2 the gradient
 * or shard region (its first 16 KB) is never read; kernel 2 may write its
 * scale row (16 bytes at offset 8 KB).  Kernel 3 sets ZERO_DEV_TIMEOUT too
 * but then quantizes its block from global memory instead, as it does on
 * any run-out wait: the bf16 values at offset 0 (2048 of them), codes at
 * 4 KB, dequantized bf16 at 8 KB, the scale at 12 KB, as zero_quant_gather
 * would write them.  Exists so that the timeout handling can be tested.     */
ZERO_API zero_status zero_debug_stream_timeout(int kernel, void* scratch, zero_dev_scalars* scalars_dev,
                                               long long timeout_ns, void* stream);

ZERO_API zero_status zero_debug_wait_timeout(zero_dev_scalars* scalars_dev, long long timeout_ns,
                                             void* stream);

/* ------------------------------------------------- allocation-free step --- */
/* The pages have no counterpart to this entry point.  It serves callers
 * that cannot allocate device memory for a workspace:
 *   - plug-ins and callbacks running inside a host framework that owns all
 *     device memory and hands them no extra buffers;
 *   - long-running services that forbid allocation once started, because a
 *     cudaMalloc may synchronise the device and its latency is unbounded;
 *   - programs whose memory budget is committed up front to a fixed pool,
 *     where a later allocation would fail.
 *
 * It is zero_step_fused with the caller's workspace replaced by one scratch
 * array that lives in the library (a file-scope __device__ array of
 * ZERO_NOALLOC_SCRATCH_BYTES = 32 KB of partial sums + 4 MB for the reduced
 * gradient; every GPU that loads the library holds it until the process
 * exits).  The call allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library routine.  The caller still passes every input and
 * output buffer.
 *   - Limit: requests whose zero_workspace_bytes(plan, hp) exceeds the
 *     scratch -- clipping with n_d > 4 and n_d*S > 2^20 parameters -- are
 *     rejected with ZERO_ERR_BOUNDS before anything is launched.  Without
 *     clipping, or with n_d <= 4, any size is accepted.
 *   - Set-up: the first call on a device (with that device current) looks up
 *     the scratch's device address, and so does the first call after a
 *     device reset (a new context may place the array elsewhere); make that
 *     first call before any stream capture.
 *   - Every call shares the one scratch array, which keeps the last call's
 *     contents; each call writes every scratch entry it reads, so nothing has
 *     to be cleared.  Calls that overlap on the GPU (other streams, other
 *     threads, other plans) race on the scratch: order them on one stream.
 * Arguments, results and errors are otherwise those of zero_step_fused.    */
#define ZERO_NOALLOC_SCRATCH_BYTES (32768u + 4u * (1u << 20))
ZERO_API zero_status zero_step_fused_noalloc(const zero_plan* plan, const zero_hparams* hp,
                                             const void* const* rank_grads, const float* master_in,
                                             const float* m_in, const float* v_in, float* master_out,
                                             float* m_out, float* v_out, void* lp_out,
                                             zero_dev_scalars* scalars_dev, void* stream);

/* Number of kernels this library has launched in this process so far (all
 * threads, all devices).  Lets a caller count the launches of a region.     */
ZERO_API unsigned long long zero_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* ZERO_H */
