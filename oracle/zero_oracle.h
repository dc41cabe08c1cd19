/*
 * zero_oracle.h -- TEST INFRASTRUCTURE ONLY.
 *
 * Declarations of the plain, slow, single-threaded CPU oracle of the ZeRO-DP
 * optimizer step.  Only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg may load this code; the product library never does.  It
 * shares no code, header, table or helper with the CUDA path.
 *
 * Sources (page title, then section):
 *   [DP-notes]  "Data parallelism and ZeRO optimization -- Hinglish notes" (6.1.8)
 *   [LLM-par]   "大模型并行技术" (LLM parallelism techniques)
 *   [itwiki]    "ZeRO (딥 러닝)"
 *   [MP-notes]  "Model parallelism (tensor, pipeline) -- Hinglish notes" (6.1.7)
 *
 * Parity unpinned: none of the functions below lacks a pin; the pins are in
 * tests/test_oracle_*.py and each names the passage or the mathematics it uses.
 */
#ifndef ZERO_ORACLE_H
#define ZERO_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ZO_BF16 0
#define ZO_FP16 1

typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
    float max_norm;     /* <= 0: no clipping                                 */
    int   loss_scaling; /* 1: dynamic loss scale with overflow skip          */
    int   scale_window; /* consecutive good steps before the scale doubles   */
    float min_scale;    /* floor of the loss scale after halving             */
} zo_hparams;

typedef struct {
    long long t;          /* committed (not skipped) steps                     */
    double beta1_pow;     /* beta1^t, repeated fp64 multiplication             */
    double beta2_pow;     /* beta2^t                                           */
    float loss_scale;     /* current loss scale (1 when loss scaling is off)   */
    int good_steps;       /* consecutive committed steps since the last change */
    int overflow;         /* 1 if the most recent step was skipped             */
    double sqnorm;        /* squared L2 norm of the averaged gradient (clip)   */
    float clip_coef;      /* coefficient applied in the most recent step       */
} zo_scalars;

/* ---- partition (flat parameter split into equal padded shards) ---- */
long long zo_shard_size(long long psi, int n_d, int shard_pad);
long long zo_valid_len(long long psi, long long shard, int r);
void zo_owner(long long j, long long shard, int* r, long long* i);

/* ---- 16-bit float encodings, written from IEEE 754 ---- */
uint16_t zo_f32_to_bf16(float x);
float zo_bf16_to_f32(uint16_t h);
uint16_t zo_f32_to_fp16(float x);
float zo_fp16_to_f32(uint16_t h);
float zo_lp_to_f32(uint16_t h, int dtype);
uint16_t zo_f32_to_lp(float x, int dtype);
void zo_f32_to_lp_array(long long n, const float* x, uint16_t* out, int dtype);
void zo_lp_to_f32_array(long long n, const uint16_t* h, float* out, int dtype);

/* ---- model-state memory and communication accounting ---- */
void zo_model_state_bytes(double psi, double n_d, int stage, double k, double out[4]);
double zo_comm_volume(int stage);

/* ---- collectives of the simulated ranks ---- */
void zo_all_reduce_mean(int n_d, long long psi, const uint16_t* const* grads, int dtype,
                        float divisor, float* out);
void zo_reduce_scatter(int n_d, long long psi, long long shard, const uint16_t* const* grads,
                       int dtype, float divisor, float* shards);
void zo_all_gather_u16(int n_d, long long psi, long long shard, const uint16_t* const* shards,
                       uint16_t* gathered);
void zo_all_gather_f32(int n_d, long long psi, long long shard, const float* const* shards,
                       float* gathered);

/* ---- Adam: textbook Adam (Kingma & Ba) in the efficient order of their
 * Section 2, decoupled weight decay as in AdamW (the pages give no equations) */
typedef struct {
    float step_size; /* lr * sqrt(1 - beta2^t) / (1 - beta1^t) */
    float eps_hat;   /* eps * sqrt(1 - beta2^t)                */
    float omb1;      /* 1 - beta1                              */
    float omb2;      /* 1 - beta2                              */
    float decay;     /* 1 - lr * weight_decay                  */
} zo_adam_consts;

void zo_adam_consts_for(const zo_hparams* hp, double beta1_pow_t, double beta2_pow_t,
                        zo_adam_consts* c);
void zo_adam_update(const zo_hparams* hp, const zo_adam_consts* c, long long n, const float* g,
                    float* p, float* m, float* v);

/* ---- clipping ---- */
double zo_sqnorm(long long n, const float* g);
float zo_clip_coef(float max_norm, double sqnorm, int* applied);

/* ---- full steps ---- */
int zo_plain_dp_step(int n_d, long long psi, const uint16_t* const* grads, int grad_dtype,
                     const zo_hparams* hp, zo_scalars* sc, float* master, float* m, float* v,
                     uint16_t* params_lp, int param_dtype);
int zo_zero_step(int n_d, long long psi, int shard_pad, int stage, const uint16_t* const* grads,
                 int grad_dtype, const zo_hparams* hp, zo_scalars* sc, float* master, float* m,
                 float* v, uint16_t* lp_shards, uint16_t* gathered, int param_dtype);
void zo_scalars_init(zo_scalars* sc, float loss_scale);

/* ---- gradient accumulation ---- */
void zo_accumulate_grads(int n_d, long long psi, const uint16_t* const* grads, int dtype,
                         const float* acc_in, float* acc_out);
int zo_zero_step_accum(int n_d, long long psi, int shard_pad, int stage, const uint16_t* const* grads,
                       int grad_dtype, const float* acc, int micro, const zo_hparams* hp, zo_scalars* sc,
                       float* master, float* m, float* v, uint16_t* lp_shards, uint16_t* gathered,
                       int param_dtype);

/* ---- block-int8 quantized gather ---- */
void zo_quantize_block(long long n, const uint16_t* x_bf16, int8_t* codes, float* scale,
                       uint16_t* deq_bf16);
void zo_quant_gather(int n_d, long long psi, long long shard, int block, const uint16_t* shards,
                     int8_t* codes, float* scales, uint16_t* gathered);

/* ---- quantized gradient exchange (ZeRO++ qgZ reading) ---- */
long long zo_qgz_rank_stride(int n_d);
void zo_quantize_ranks(int n_d, long long psi, long long shard, int block, const uint16_t* const* grads,
                       int8_t* const* codes, float* scales);
void zo_reduce_scatter_q(int n_d, long long psi, long long shard, int block, const int8_t* const* codes,
                         const float* scales, float divisor, float* shards);
void zo_reduce_points_q(int n_d, long long n, const int8_t* const* codes, const float* const* scales,
                        float divisor, float* out);
int zo_zero_step_qgz(int n_d, long long psi, int shard_pad, int stage, int block, const int8_t* const* codes,
                     const float* scales, const zo_hparams* hp, zo_scalars* sc, float* master, float* m,
                     float* v, uint16_t* lp_shards, uint16_t* gathered, int param_dtype);

#ifdef __cplusplus
}
#endif
#endif
