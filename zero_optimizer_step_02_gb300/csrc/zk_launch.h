// zk_launch.h -- host-side launch interface of the libzero kernels.
#pragma once

#include <cuda_runtime.h>

#include "zero.h"

namespace zk {

enum {
    OP_FUSED = 0,
    OP_REDUCE = 1,
    OP_ADAM = 2,
    OP_QFUSED = 3,  // fused step + int8 gather epilogue
    OP_QADAM = 4    // Adam from an fp32 reduced gradient + int8 gather epilogue
};

// rank streams that carry int8 codes with per-rank fp32 block scales (the
// quantized gradient exchange) instead of bf16 / fp16 values
constexpr int kGradQ8 = 2;

// Arguments of one launch of the streaming engine (kernel parameter space).
//
// Tiles: element ranges of 2048 laid over "segments".  A flat launch has one
// segment [base, limit); a per-shard launch (fused quantized gather) has n_seg
// segments starting at base + s * seg_stride, each seg_len long and clipped
// at limit (= Psi), so that no tile crosses a shard boundary.
struct StreamArgs {
    const void* rank[ZERO_MAX_RANKS];  // 16-bit gradient buffers, rank order
    const float* side[4];              // fp32 inputs: OP_FUSED/OP_QFUSED {master, m, v, carry};
                                       // OP_ADAM/OP_QADAM {g, master, m, v}; OP_REDUCE {carry}
                                       // (carry: F_CARRY only)
    float* out_f32[3];                 // OP_FUSED/OP_ADAM/OP_QFUSED/OP_QADAM {master, m, v}; OP_REDUCE {g or null}
    void* out_lp;                      // 16-bit parameters out (null: none)
    const float* q_rank_scales;        // kGradQ8 ranks: scales, block-major, rank-minor:
    long long q_rank_scale_stride;     //   [(shard * blocks_per_shard + block) * stride + rank], stride % 4 == 0
    signed char* q_codes;              // fused quantized gather (F_QUANT)
    float* q_scales;
    void* q_gathered;
    zero_dev_scalars* sc;
    double* partials;                  // OP_REDUCE + F_SQNORM: one fp64 per CTA
    const double* fin_partials;        // F_FINALIZE: the reduce pass's partials ...
    int fin_n;                         // ... and how many
    long long base, seg_stride, seg_len, limit, tiles_per_seg, q_blocks_per_shard;
    int n_seg;
    int n_ranks;                       // rank streams (0 for OP_ADAM and OP_QADAM)
    int micro;                         // micro-batches in the mean (divisor n_ranks * micro); 0 reads as 1
    int n_side;                        // fp32 side streams
    int n_side_tma;                    // the first n_side_tma of them are staged by bulk copies; the
                                       // rest (state in page-locked host memory) are read directly
    int tma_ok;                        // every full tile is 16-byte aligned in every stream
    int flags;                         // F_* of zk_common.cuh
    int stages;                        // set by the launcher
    unsigned stage_bytes;              // set by the launcher
    int grid;                          // set by the launcher
    unsigned long long timeout_ns;
    zero_hparams hp;
};

cudaError_t launch_stream(int op, int grad_dtype, int param_dtype, StreamArgs& a, cudaStream_t st);

// Arguments of the small-problem fused step (zk_small.cu): the plain fused
// step over [lo, hi) (lo a multiple of 4), state in device memory.
struct SmallArgs {
    const void* rank[ZERO_MAX_RANKS];  // 16-bit gradient buffers, rank order
    const float* master_in;
    const float* m_in;
    const float* v_in;
    float* master_out;
    float* m_out;
    float* v_out;
    void* lp_out;                      // 16-bit parameters out (null: none)
    zero_dev_scalars* sc;
    long long lo, hi;
    int n_ranks;
    int epilogue;                      // the last CTA commits the step scalars
    zero_hparams hp;
};

// true when n elements would give the streaming engine under two tiles per SM
bool small_step_fits(long long n);
cudaError_t launch_small_step(int grad_dtype, int param_dtype, const SmallArgs& a, cudaStream_t st);

// every kernel launch of the library adds one (zero_launch_count)
void count_launch();
unsigned long long launch_count();

// auxiliary kernels (zk_aux.cu)
cudaError_t launch_scalars_init(zero_dev_scalars* sc, float loss_scale, cudaStream_t st);
cudaError_t launch_finalize_sqnorm(const double* partials, int n, const zero_hparams& hp,
                                   zero_dev_scalars* sc, cudaStream_t st);
cudaError_t launch_sqnorm_f32(const float* g, long long n, double* partials, int* n_partials,
                              cudaStream_t st);
cudaError_t launch_epilogue(const zero_hparams& hp, zero_dev_scalars* sc, cudaStream_t st);
cudaError_t launch_repair(const float* master_in, const float* m_in, const float* v_in, float* master_out,
                          float* m_out, float* v_out, void* lp_out, int param_dtype, long long psi, zero_dev_scalars* sc,
                          cudaStream_t st);
// starve: issue no copy, so every wait runs out (tests the timeout path)
cudaError_t launch_all_gather(const void* const* shards, int n_d, long long shard, long long psi,
                              void* gathered, zero_dev_scalars* sc, cudaStream_t st, bool starve = false);
// sc may be null (a wait that runs out is then not reported; the results are
// complete either way); starve: issue no copy, so every wait runs out and the
// blocks are read from global memory (tests that path)
cudaError_t launch_quant_gather(const void* shards, int n_d, long long shard, long long psi,
                                int block, signed char* codes, float* scales, void* gathered,
                                zero_dev_scalars* sc, cudaStream_t st, bool starve = false);
cudaError_t launch_quantize_grads(const void* const* ranks, int n_d, long long shard, long long psi, int block,
                                  signed char* const* codes, float* scales, zero_dev_scalars* sc, cudaStream_t st,
                                  bool starve = false);
cudaError_t launch_debug_wait(zero_dev_scalars* sc, unsigned long long timeout_ns, cudaStream_t st);

}  // namespace zk
