// zk_capi.cu -- the C ABI of libzero.so: plans, argument checks, and the pass
// schedules of the ZeRO-DP step.  Declarations and the contract of every
// entry point are in include/zero.h.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>

#include <nvtx3/nvToolsExt.h>

#include "zk_common.cuh"
#include "zk_launch.h"

struct zero_plan {
    long long psi;
    int n_d;
    int stage;
    int grad_dtype;
    int param_dtype;
    int shard_pad;
    long long shard;   // S
    long long padded;  // n_d * S
    long long bucket;  // elements per fused-step bucket (multiple of the tile)
};

namespace {

using zk::StreamArgs;

// An NVTX range named after the entry point around each call that launches
// work, so that profilers (nsys, ncu --nvtx) group its kernels; with no tool
// attached it costs a branch.
struct CallRange {
    explicit CallRange(const char* name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
    CallRange(const CallRange&) = delete;
    CallRange& operator=(const CallRange&) = delete;
};
#define ZK_CALL_RANGE() const CallRange zk_call_range_(__func__)

constexpr size_t kPartialBytes = sizeof(double) * zk::kMaxPartials;  // 32 KB, 256-aligned

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

zero_status from_cuda(cudaError_t e) { return e == cudaSuccess ? ZERO_OK : ZERO_ERR_CUDA; }

#define ZK_TRY(expr)                              \
    do {                                          \
        const cudaError_t e_ = (expr);            \
        if (e_ != cudaSuccess) return ZERO_ERR_CUDA; \
    } while (0)

zero_status check_hparams(const zero_hparams* hp)
{
    if (hp == nullptr) return ZERO_ERR_INVALID_ARG;
    const float v[] = {hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay, hp->max_norm};
    for (float x : v)
        if (std::isnan(x)) return ZERO_ERR_INVALID_ARG;
    if (hp->beta1 < 0.0f || hp->beta1 >= 1.0f || hp->beta2 < 0.0f || hp->beta2 >= 1.0f) return ZERO_ERR_INVALID_ARG;
    if (hp->lr < 0.0f || hp->eps < 0.0f || hp->weight_decay < 0.0f) return ZERO_ERR_INVALID_ARG;
    if (hp->loss_scaling != 0 && hp->loss_scaling != 1) return ZERO_ERR_INVALID_ARG;
    if (hp->loss_scaling && (hp->scale_window < 1 || !(hp->min_scale > 0.0f))) return ZERO_ERR_INVALID_ARG;
    return ZERO_OK;
}

zero_status check_ranks(const zero_plan* p, const void* const* ranks)
{
    if (ranks == nullptr) return ZERO_ERR_INVALID_ARG;
    for (int r = 0; r < p->n_d; ++r) {
        if (ranks[r] == nullptr) return ZERO_ERR_INVALID_ARG;
        if (!aligned(ranks[r], 16)) return ZERO_ERR_MISALIGNED;
    }
    return ZERO_OK;
}

zero_status check_dev(const void* ptr, uintptr_t align = 16)
{
    if (ptr == nullptr) return ZERO_ERR_INVALID_ARG;
    return aligned(ptr, align) ? ZERO_OK : ZERO_ERR_MISALIGNED;
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

long long tiles_of(long long n) { return (n + zk::kTile - 1) / zk::kTile; }

// flat tile map over [lo, hi)
void set_flat(StreamArgs& a, long long lo, long long hi)
{
    a.base = lo;
    a.seg_stride = 0;
    a.seg_len = hi - lo;
    a.limit = hi;
    a.n_seg = 1;
    a.tiles_per_seg = tiles_of(hi - lo);
    a.tma_ok = (lo % 8) == 0 ? 1 : 0;
}

StreamArgs base_args(const zero_hparams* hp, zero_dev_scalars* sc)
{
    StreamArgs a;
    std::memset(&a, 0, sizeof(a));
    a.sc = sc;
    a.timeout_ns = zk::kDefaultTimeoutNs;
    if (hp != nullptr) a.hp = *hp;
    return a;
}

void set_ranks(StreamArgs& a, const zero_plan* p, const void* const* ranks)
{
    a.n_ranks = p->n_d;
    for (int r = 0; r < p->n_d; ++r) a.rank[r] = ranks[r];
}

double* partials_of(void* ws) { return static_cast<double*>(ws); }
float* ghat_of(void* ws) { return reinterpret_cast<float*>(static_cast<char*>(ws) + kPartialBytes); }

// the reduced gradient goes through HBM only when that moves fewer bytes than
// reading the rank gradients twice: 4 + 4 bytes against 2 * n_d
bool clip_materialises(const zero_plan* p) { return p->n_d > 4; }

// grid the streaming launch uses for a flat range of n elements (the partial
// sums of a reduce are one per CTA; zero_grad_sqnorm recomputes this count)
int reduce_grid(long long n)
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    long long g = tiles_of(n);
    if (g > sms) g = sms;
    if (g > zk::kMaxPartials) g = zk::kMaxPartials;
    return static_cast<int>(g);
}

// Gradient accumulation: carry (fp32, indexed like the gradients) is added to
// the rank sum, and the mean divides by n_d * micro.
struct Accum {
    const float* carry;
    int micro;
};
constexpr Accum kNoAccum = {nullptr, 1};

void set_accum(StreamArgs& a, const Accum& acc, int slot)
{
    a.micro = acc.micro;
    if (acc.carry == nullptr) return;
    a.side[slot] = acc.carry;
    a.n_side = slot + 1;
    a.flags |= zk::F_CARRY;
}

// One reduce pass over [0, psi): optional fp32 output, squared-norm partials,
// non-finite detection in loss-scaling mode.
zero_status run_reduce(const zero_plan* p, const zero_hparams* hp, const void* const* ranks, float* out,
                       bool sqnorm, void* ws, zero_dev_scalars* sc, cudaStream_t st, int* grid_out = nullptr,
                       const Accum& acc = kNoAccum)
{
    StreamArgs a = base_args(hp, sc);
    set_ranks(a, p, ranks);
    set_flat(a, 0, p->psi);
    a.n_side = 0;
    a.out_f32[0] = out;
    a.partials = sqnorm ? partials_of(ws) : nullptr;
    a.flags = (sqnorm ? zk::F_SQNORM : 0) | (hp->loss_scaling ? (zk::F_DETECT | zk::F_LSCALE) : 0);
    set_accum(a, acc, 0);
    if (out != nullptr && !aligned(out, 16)) a.tma_ok = 0;
    const zero_status s = from_cuda(zk::launch_stream(zk::OP_REDUCE, p->grad_dtype, p->param_dtype, a, st));
    if (grid_out != nullptr) *grid_out = a.grid;
    return s;
}

// F_FINALIZE inputs: the partial sums a reduce pass left in the workspace
void set_finalize(StreamArgs& a, void* ws, int n)
{
    a.fin_partials = partials_of(ws);
    a.fin_n = n;
}

// flags may hold F_EPILOGUE (given to the last bucket only) and F_FINALIZE
// (fin_ws / fin_n: the partials of the preceding reduce pass)
zero_status run_fused(const zero_plan* p, const zero_hparams* hp, const void* const* ranks, const float* mi,
                      const float* m_in, const float* vi, float* mo, float* m_out, float* vo, void* lp,
                      int flags, zero_dev_scalars* sc, cudaStream_t st, void* fin_ws = nullptr, int fin_n = 0,
                      bool host_state = false, const Accum& acc = kNoAccum)
{
    // buckets only when no global check ties the pieces together
    const long long step =
        (flags & (zk::F_CLIP | zk::F_GUARD | zk::F_DETECT | zk::F_FINALIZE)) ? p->psi : p->bucket;
    for (long long lo = 0; lo < p->psi; lo += step) {
        const long long hi = lo + step < p->psi ? lo + step : p->psi;
        // a plain step too small to fill the engine's pipeline: the small-problem kernel
        if ((flags & ~zk::F_EPILOGUE) == 0 && !host_state && acc.carry == nullptr && zk::small_step_fits(hi - lo)) {
            zk::SmallArgs b;
            std::memset(&b, 0, sizeof(b));
            for (int r = 0; r < p->n_d; ++r) b.rank[r] = ranks[r];
            b.master_in = mi;
            b.m_in = m_in;
            b.v_in = vi;
            b.master_out = mo;
            b.m_out = m_out;
            b.v_out = vo;
            b.lp_out = lp;
            b.sc = sc;
            b.lo = lo;
            b.hi = hi;
            b.n_ranks = p->n_d;
            b.epilogue = (hi == p->psi && (flags & zk::F_EPILOGUE)) ? 1 : 0;
            b.hp = *hp;
            const zero_status s = from_cuda(zk::launch_small_step(p->grad_dtype, p->param_dtype, b, st));
            if (s != ZERO_OK) return s;
            continue;
        }
        StreamArgs a = base_args(hp, sc);
        if (flags & zk::F_FINALIZE) set_finalize(a, fin_ws, fin_n);
        set_ranks(a, p, ranks);
        set_flat(a, lo, hi);
        a.n_side = 3;
        a.n_side_tma = host_state ? 0 : 3;
        a.side[0] = mi;
        a.side[1] = m_in;
        a.side[2] = vi;
        a.out_f32[0] = mo;
        a.out_f32[1] = m_out;
        a.out_f32[2] = vo;
        a.out_lp = lp;
        a.flags = (hi == p->psi ? flags : (flags & ~zk::F_EPILOGUE)) | (host_state ? zk::F_HOST_STATE : 0);
        set_accum(a, acc, 3);   // the carry is read directly, never staged
        const zero_status s = from_cuda(zk::launch_stream(zk::OP_FUSED, p->grad_dtype, p->param_dtype, a, st));
        if (s != ZERO_OK) return s;
    }
    return ZERO_OK;
}

zero_status run_adam(const zero_plan* p, const zero_hparams* hp, const float* g, const float* mi,
                     const float* m_in, const float* vi, float* mo, float* m_out, float* vo, void* lp, int flags,
                     zero_dev_scalars* sc, cudaStream_t st, void* fin_ws = nullptr, int fin_n = 0,
                     bool host_state = false)
{
    StreamArgs a = base_args(hp, sc);
    if (flags & zk::F_FINALIZE) set_finalize(a, fin_ws, fin_n);
    set_flat(a, 0, p->psi);
    a.n_ranks = 0;
    a.n_side = 4;
    a.n_side_tma = host_state ? 1 : 4;   // the reduced gradient stays in HBM
    a.side[0] = g;
    a.side[1] = mi;
    a.side[2] = m_in;
    a.side[3] = vi;
    a.out_f32[0] = mo;
    a.out_f32[1] = m_out;
    a.out_f32[2] = vo;
    a.out_lp = lp;
    a.flags = flags | (host_state ? zk::F_HOST_STATE : 0);
    return from_cuda(zk::launch_stream(zk::OP_ADAM, p->grad_dtype, p->param_dtype, a, st));
}

// int8 rank streams (the quantized gradient exchange): tiles inside shards,
// so that every 2048-element block of a tile has one scale per rank
void set_q8_ranks(StreamArgs& a, const zero_plan* p, const signed char* const* codes, const float* scales)
{
    a.n_ranks = p->n_d;
    for (int r = 0; r < p->n_d; ++r) a.rank[r] = codes[r];
    a.base = 0;
    a.seg_stride = p->shard;
    a.seg_len = p->shard;
    a.limit = p->psi;
    a.n_seg = p->n_d;
    a.tiles_per_seg = tiles_of(p->shard);
    a.q_blocks_per_shard = (p->shard + zk::kQuantBlock - 1) / zk::kQuantBlock;
    a.q_rank_scales = scales;
    a.q_rank_scale_stride = (p->n_d + 3) / 4 * 4;
    a.tma_ok = (p->shard % 16) == 0 ? 1 : 0;   // int8 slices start 16-byte aligned
}

// reduce pass over int8 ranks: squared-norm partials, optional fp32 output
zero_status run_reduce_q8(const zero_plan* p, const zero_hparams* hp, const signed char* const* codes,
                          const float* scales, float* out, void* ws, zero_dev_scalars* sc, cudaStream_t st,
                          int* grid_out)
{
    StreamArgs a = base_args(hp, sc);
    set_q8_ranks(a, p, codes, scales);
    a.n_side = 0;
    a.out_f32[0] = out;
    a.partials = partials_of(ws);
    a.flags = zk::F_SQNORM;
    const zero_status s = from_cuda(zk::launch_stream(zk::OP_REDUCE, zk::kGradQ8, p->param_dtype, a, st));
    *grid_out = a.grid;
    return s;
}

// the fused step over int8 ranks (flags: F_EPILOGUE, and F_CLIP | F_FINALIZE
// after a reduce pass whose partials are in ws)
zero_status run_fused_q8(const zero_plan* p, const zero_hparams* hp, const signed char* const* codes,
                         const float* scales, const float* mi, const float* m_in, const float* vi, float* mo,
                         float* m_out, float* vo, void* lp, int flags, zero_dev_scalars* sc, cudaStream_t st,
                         void* fin_ws = nullptr, int fin_n = 0)
{
    StreamArgs a = base_args(hp, sc);
    if (flags & zk::F_FINALIZE) set_finalize(a, fin_ws, fin_n);
    set_q8_ranks(a, p, codes, scales);
    a.n_side = 3;
    // a full stage of int8 ranks or more (N_d >= 16, one or several rank groups
    // per tile): the state is read with direct 16-byte loads instead of being
    // staged, so the stages hold codes only and the ring gets three of them
    // (N_d = 64: 3.93 -> 3.55 ms, 92% -> 102% of the copy rate; N_d = 32: 2.26
    // -> 2.18 ms; N_d = 16: 1.69 -> 1.67 ms).  With fewer ranks the loads' latency
    // is not hidden (N_d = 8: 1.37 -> 1.69 ms), and the 16-bit fused step
    // measured slower that way at any N_d (16: 2.16 -> 2.22 ms): both keep the
    // state staged.
    a.n_side_tma = p->n_d >= 2 * zk::kGroupRanks ? 0 : 3;
    a.side[0] = mi;
    a.side[1] = m_in;
    a.side[2] = vi;
    a.out_f32[0] = mo;
    a.out_f32[1] = m_out;
    a.out_f32[2] = vo;
    a.out_lp = lp;
    a.flags = flags;
    return from_cuda(zk::launch_stream(zk::OP_FUSED, zk::kGradQ8, p->param_dtype, a, st));
}

// two arrays of n bytes share a byte
// Adam from the fp32 reduced gradient g with the int8 gather as its epilogue
// (tiles inside shards: each 2048-element block starts in its shard); flags
// hold F_QUANT | F_EPILOGUE and F_CLIP | F_FINALIZE (the partials in ws) and
// F_GUARD as the schedule needs
zero_status run_qadam(const zero_plan* p, const zero_hparams* hp, const float* g, const float* mi,
                      const float* m_in, const float* vi, float* mo, float* m_out, float* vo, signed char* codes,
                      float* scales, void* gathered, int flags, zero_dev_scalars* sc, cudaStream_t st, void* fin_ws,
                      int fin_n)
{
    StreamArgs a = base_args(hp, sc);
    if (flags & zk::F_FINALIZE) set_finalize(a, fin_ws, fin_n);
    a.n_ranks = 0;
    a.base = 0;
    a.seg_stride = p->shard;
    a.seg_len = p->shard;
    a.limit = p->psi;
    a.n_seg = p->n_d;
    a.tiles_per_seg = tiles_of(p->shard);
    a.q_blocks_per_shard = (p->shard + zk::kQuantBlock - 1) / zk::kQuantBlock;
    a.tma_ok = (p->shard % 4) == 0 ? 1 : 0;   // every fp32 stream of a tile starts 16-byte aligned
    a.n_side = 4;
    a.n_side_tma = 4;
    a.side[0] = g;
    a.side[1] = mi;
    a.side[2] = m_in;
    a.side[3] = vi;
    a.out_f32[0] = mo;
    a.out_f32[1] = m_out;
    a.out_f32[2] = vo;
    a.q_codes = codes;
    a.q_scales = scales;
    a.q_gathered = gathered;
    a.flags = flags;
    return from_cuda(zk::launch_stream(zk::OP_QADAM, ZERO_BF16, p->param_dtype, a, st));
}

// page-locked host memory the device reaches at the same address (state kept
// in host memory); anything else is refused before a launch
bool host_mapped(const void* q)
{
    if (q == nullptr) return false;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, q) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeHost && at.devicePointer == q;
}

bool overlaps(const void* a, const void* b, uintptr_t n)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + n && y < x + n;
}

// master/m/v in and out, n_d*S floats each: out may equal in, array by array,
// but all three or none; no output shares a byte with another output, nor
// with an input other than its own
zero_status check_state(const zero_plan* p, const float* mi, const float* m_in, const float* vi, float* mo,
                        float* m_out, float* vo)
{
    const void* ptrs[] = {mi, m_in, vi, mo, m_out, vo};
    for (const void* q : ptrs) {
        const zero_status s = check_dev(q);
        if (s != ZERO_OK) return s;
    }
    const int alias = (mo == mi) + (m_out == m_in) + (vo == vi);
    if (alias != 0 && alias != 3) return ZERO_ERR_INVALID_ARG;
    const uintptr_t n = sizeof(float) * static_cast<uintptr_t>(p->padded);
    const void* outs[3] = {mo, m_out, vo};
    const void* ins[3] = {mi, m_in, vi};
    for (int i = 0; i < 3; ++i)
        for (int j = 0; j < 3; ++j) {
            if (i != j && overlaps(outs[i], outs[j], n)) return ZERO_ERR_INVALID_ARG;
            if ((i != j || alias == 0) && overlaps(outs[i], ins[j], n)) return ZERO_ERR_INVALID_ARG;
        }
    return ZERO_OK;
}

}  // namespace

extern "C" {

ZERO_API const char* zero_status_str(zero_status s)
{
    switch (s) {
    case ZERO_OK: return "ok";
    case ZERO_ERR_INVALID_ARG: return "invalid argument";
    case ZERO_ERR_MISALIGNED: return "misaligned device pointer";
    case ZERO_ERR_UNSUPPORTED: return "unsupported request";
    case ZERO_ERR_CUDA: return "CUDA error";
    case ZERO_ERR_TIMEOUT: return "device wait timed out";
    case ZERO_ERR_BOUNDS: return "request exceeds a fixed capacity";
    }
    return "unknown status";
}

ZERO_API int zero_abi_version(void) { return ZERO_ABI_VERSION; }

ZERO_API size_t zero_dev_scalars_size(void) { return sizeof(zero_dev_scalars); }

ZERO_API zero_status zero_plan_create_ex(zero_plan** out, long long psi, int n_d, int stage, zero_dtype grad_dtype,
                                         int shard_pad, const zero_plan_opts* opts)
{
    if (out == nullptr) return ZERO_ERR_INVALID_ARG;
    *out = nullptr;
    if (psi < 1 || n_d < 1 || n_d > ZERO_MAX_RANKS || stage < 1 || stage > 3) return ZERO_ERR_INVALID_ARG;
    if (shard_pad < 1 || shard_pad > ZERO_MAX_SHARD_PAD) return ZERO_ERR_INVALID_ARG;
    if (grad_dtype != ZERO_BF16 && grad_dtype != ZERO_FP16) return ZERO_ERR_INVALID_ARG;
    int pdt = ZERO_BF16;
    long long bucket = 0;
    if (opts != nullptr) {
        if (opts->param_dtype_set) {
            if (opts->param_dtype != ZERO_BF16 && opts->param_dtype != ZERO_FP16) return ZERO_ERR_INVALID_ARG;
            pdt = opts->param_dtype;
        }
        bucket = opts->reduce_bucket_elems;
    }
    if (psi > (1LL << 40)) return ZERO_ERR_INVALID_ARG;
    zero_plan* p = new (std::nothrow) zero_plan;
    if (p == nullptr) return ZERO_ERR_BOUNDS;
    p->psi = psi;
    p->n_d = n_d;
    p->stage = stage;
    p->grad_dtype = grad_dtype;
    p->param_dtype = pdt;
    p->shard_pad = shard_pad;
    const long long per_rank = (psi + n_d - 1) / n_d;
    p->shard = (per_rank + shard_pad - 1) / shard_pad * shard_pad;
    p->padded = p->shard * n_d;
    if (bucket <= 0 || bucket >= psi) {
        p->bucket = psi;
    } else {
        p->bucket = (bucket + zk::kTile - 1) / zk::kTile * zk::kTile;
    }
    *out = p;
    return ZERO_OK;
}

ZERO_API zero_status zero_plan_create(zero_plan** out, long long psi, int n_d, int stage, zero_dtype grad_dtype,
                                      int shard_pad)
{
    return zero_plan_create_ex(out, psi, n_d, stage, grad_dtype, shard_pad, nullptr);
}

ZERO_API void zero_plan_destroy(zero_plan* plan) { delete plan; }

ZERO_API zero_status zero_plan_query(const zero_plan* p, long long* shard_size, long long* padded_psi,
                                     long long* valid_len)
{
    if (p == nullptr) return ZERO_ERR_INVALID_ARG;
    if (shard_size) *shard_size = p->shard;
    if (padded_psi) *padded_psi = p->padded;
    if (valid_len) {
        for (int r = 0; r < p->n_d; ++r) {
            long long v = p->psi - static_cast<long long>(r) * p->shard;
            valid_len[r] = v < 0 ? 0 : (v > p->shard ? p->shard : v);
        }
    }
    return ZERO_OK;
}

ZERO_API zero_status zero_plan_memory(const zero_plan* p, int stage, double k, double bytes_out[4])
{
    if (p == nullptr || bytes_out == nullptr || stage < 0 || stage > 3 || !(k >= 0.0)) return ZERO_ERR_INVALID_ARG;
    const double psi = static_cast<double>(p->psi), n = static_cast<double>(p->n_d);
    // which of the three model states are divided among the ranks at this stage
    const bool part_opt = stage >= 1, part_grad = stage >= 2, part_param = stage >= 3;
    bytes_out[0] = part_param ? 2.0 * psi / n : 2.0 * psi;
    bytes_out[1] = part_grad ? 2.0 * psi / n : 2.0 * psi;
    bytes_out[2] = part_opt ? k * psi / n : k * psi;
    bytes_out[3] = bytes_out[0] + bytes_out[1] + bytes_out[2];
    return ZERO_OK;
}

ZERO_API zero_status zero_plan_comm_volume(const zero_plan* p, int stage, double* elems_out)
{
    if (p == nullptr || elems_out == nullptr || stage < 0 || stage > 3) return ZERO_ERR_INVALID_ARG;
    const int gathers = stage == 3 ? 2 : 1;  // forward and backward gathers in stage 3
    *elems_out = static_cast<double>(p->psi) * (1 + gathers);
    return ZERO_OK;
}

ZERO_API size_t zero_workspace_bytes(const zero_plan* p, const zero_hparams* hp)
{
    if (p == nullptr) return 0;
    size_t bytes = kPartialBytes;
    if (hp != nullptr && hp->max_norm > 0.0f && clip_materialises(p)) bytes += sizeof(float) * static_cast<size_t>(p->padded);
    return bytes;
}

ZERO_API zero_status zero_scalars_init(zero_dev_scalars* sc, float loss_scale, void* stream)
{
    ZK_CALL_RANGE();
    const zero_status s = check_dev(sc, 256);
    if (s != ZERO_OK) return s;
    if (!(loss_scale > 0.0f) || std::isinf(loss_scale)) return ZERO_ERR_INVALID_ARG;
    return from_cuda(zk::launch_scalars_init(sc, loss_scale, as_stream(stream)));
}

ZERO_API zero_status zero_reduce_scatter(const zero_plan* p, const void* const* ranks, const zero_hparams* hp,
                                         zero_dev_scalars* sc, float* grad_shards, void* ws, void* stream)
{
    ZK_CALL_RANGE();
    if (p == nullptr) return ZERO_ERR_INVALID_ARG;
    zero_status s;
    if ((s = check_hparams(hp)) != ZERO_OK) return s;
    if ((s = check_ranks(p, ranks)) != ZERO_OK) return s;
    if ((s = check_dev(sc, 256)) != ZERO_OK) return s;
    if ((s = check_dev(grad_shards)) != ZERO_OK) return s;
    if ((s = check_dev(ws, 256)) != ZERO_OK) return s;
    const cudaStream_t st = as_stream(stream);
    if ((s = run_reduce(p, hp, ranks, grad_shards, true, ws, sc, st)) != ZERO_OK) return s;
    if (p->padded > p->psi)
        ZK_TRY(cudaMemsetAsync(grad_shards + p->psi, 0, sizeof(float) * static_cast<size_t>(p->padded - p->psi), st));
    return ZERO_OK;
}

ZERO_API zero_status zero_grad_sqnorm(const zero_plan* p, const float* grad_shards, const zero_hparams* hp,
                                      zero_dev_scalars* sc, void* ws, void* stream)
{
    ZK_CALL_RANGE();
    if (p == nullptr) return ZERO_ERR_INVALID_ARG;
    zero_status s;
    if ((s = check_hparams(hp)) != ZERO_OK) return s;
    if ((s = check_dev(sc, 256)) != ZERO_OK) return s;
    if ((s = check_dev(ws, 256)) != ZERO_OK) return s;
    const cudaStream_t st = as_stream(stream);
    int n = 0;
    if (grad_shards != nullptr) {
        if (!aligned(grad_shards, 16)) return ZERO_ERR_MISALIGNED;
        ZK_TRY(zk::launch_sqnorm_f32(grad_shards, p->psi, partials_of(ws), &n, st));
    } else {
        n = reduce_grid(p->psi);
        if (n <= 0) return ZERO_ERR_CUDA;
    }
    return from_cuda(zk::launch_finalize_sqnorm(partials_of(ws), n, *hp, sc, st));
}

ZERO_API zero_status zero_adam_shard_step(const zero_plan* p, const zero_hparams* hp, const float* grad_shards,
                                          float* master, float* m, float* v, void* lp_out, zero_dev_scalars* sc,
                                          void* stream)
{
    ZK_CALL_RANGE();
    if (p == nullptr) return ZERO_ERR_INVALID_ARG;
    zero_status s;
    if ((s = check_hparams(hp)) != ZERO_OK) return s;
    if ((s = check_dev(sc, 256)) != ZERO_OK) return s;
    if ((s = check_dev(grad_shards)) != ZERO_OK) return s;
    if ((s = check_state(p, master, m, v, master, m, v)) != ZERO_OK) return s;
    if (lp_out != nullptr && !aligned(lp_out, 16)) return ZERO_ERR_MISALIGNED;
    const cudaStream_t st = as_stream(stream);
    const int flags =
        (hp->max_norm > 0.0f ? zk::F_CLIP : 0) | (hp->loss_scaling ? zk::F_GUARD : 0) | zk::F_EPILOGUE;
    return run_adam(p, hp, grad_shards, master, m, v, master, m, v, lp_out, flags, sc, st);
}

ZERO_API zero_status zero_all_gather(const zero_plan* p, const void* const* shards, void* gathered,
                                     zero_dev_scalars* sc, void* stream)
{
    ZK_CALL_RANGE();
    if (p == nullptr || shards == nullptr) return ZERO_ERR_INVALID_ARG;
    // shard pointers need only element (2-byte) alignment: shards cut from one
    // flat buffer at an odd S are legal; the bulk-copy ring is used when all
    // of them are 16-byte aligned and S is a multiple of 8
    for (int r = 0; r < p->n_d; ++r) {
        if (shards[r] == nullptr) return ZERO_ERR_INVALID_ARG;
        if (!aligned(shards[r], 2)) return ZERO_ERR_MISALIGNED;
    }
    zero_status s;
    if ((s = check_dev(gathered)) != ZERO_OK) return s;
    if (sc != nullptr && !aligned(sc, 256)) return ZERO_ERR_MISALIGNED;
    return from_cuda(zk::launch_all_gather(shards, p->n_d, p->shard, p->psi, gathered, sc, as_stream(stream)));
}

namespace {

// The pass schedules of the fused step.  host_state: master/m/v live in
// page-locked host memory and are read and written directly by the kernels.
zero_status fused_step(const zero_plan* p, const zero_hparams* hp, const void* const* ranks, const float* mi,
                       const float* m_in, const float* vi, float* mo, float* m_out, float* vo, void* lp,
                       zero_dev_scalars* sc, void* ws, void* stream, bool host_state, const Accum& acc = kNoAccum)
{
    if (p == nullptr) return ZERO_ERR_INVALID_ARG;
    zero_status s;
    if ((s = check_hparams(hp)) != ZERO_OK) return s;
    if ((s = check_ranks(p, ranks)) != ZERO_OK) return s;
    if ((s = check_dev(sc, 256)) != ZERO_OK) return s;
    if ((s = check_state(p, mi, m_in, vi, mo, m_out, vo)) != ZERO_OK) return s;
    if (lp != nullptr && !aligned(lp, 16)) return ZERO_ERR_MISALIGNED;
    const bool clip = hp->max_norm > 0.0f;
    const bool ls = hp->loss_scaling != 0;
    const bool inplace = mo == mi;
    if ((clip || ls) && (s = check_dev(ws, 256)) != ZERO_OK) return s;
    const cudaStream_t st = as_stream(stream);
    const int lsf = ls ? zk::F_LSCALE : 0;
    // the kernel that ends the step commits the scalars itself (F_EPILOGUE),
    // except when a repair pass still has to read the step's overflow flag
    const bool speculative = ls && !inplace;
    const int epi = speculative ? 0 : zk::F_EPILOGUE;

    if (!clip) {
        if (!ls) {
            if ((s = run_fused(p, hp, ranks, mi, m_in, vi, mo, m_out, vo, lp, epi, sc, st, nullptr, 0, host_state, acc)) != ZERO_OK) return s;
        } else if (speculative) {
            // update while detecting; undo from the in state if flagged
            if ((s = run_fused(p, hp, ranks, mi, m_in, vi, mo, m_out, vo, lp, zk::F_DETECT | lsf, sc, st, nullptr, 0, host_state, acc)) != ZERO_OK) return s;
        } else {
            // in place: a read-only check pass first, then the guarded update
            if ((s = run_reduce(p, hp, ranks, nullptr, false, ws, sc, st, nullptr, acc)) != ZERO_OK) return s;
            if ((s = run_fused(p, hp, ranks, mi, m_in, vi, mo, m_out, vo, lp, zk::F_GUARD | lsf | epi, sc, st, nullptr, 0, host_state, acc)) != ZERO_OK) return s;
        }
    } else {
        // the update kernel finishes the reduce pass's norm in its prologue
        const int guard = ls ? zk::F_GUARD : 0;
        int n = 0;
        if (clip_materialises(p)) {
            float* g = ghat_of(ws);
            if ((s = run_reduce(p, hp, ranks, g, true, ws, sc, st, &n, acc)) != ZERO_OK) return s;
            // the Adam pass walks the tiles from the end: the reduced gradient the
            // reduce pass wrote last is still in L2
            if ((s = run_adam(p, hp, g, mi, m_in, vi, mo, m_out, vo, lp,
                              zk::F_CLIP | zk::F_FINALIZE | guard | epi | zk::F_REVERSE, sc, st, ws, n, host_state)) != ZERO_OK)
                return s;
        } else {
            if ((s = run_reduce(p, hp, ranks, nullptr, true, ws, sc, st, &n, acc)) != ZERO_OK) return s;
            if ((s = run_fused(p, hp, ranks, mi, m_in, vi, mo, m_out, vo, lp,
                               zk::F_CLIP | zk::F_FINALIZE | guard | lsf | epi, sc, st, ws, n, host_state, acc)) != ZERO_OK)
                return s;
        }
    }
    if (!speculative) return ZERO_OK;
    ZK_TRY(zk::launch_repair(mi, m_in, vi, mo, m_out, vo, lp, p->param_dtype, p->psi, sc, st));
    return from_cuda(zk::launch_epilogue(*hp, sc, st));
}

}  // namespace

ZERO_API zero_status zero_step_fused(const zero_plan* p, const zero_hparams* hp, const void* const* ranks,
                                     const float* mi, const float* m_in, const float* vi, float* mo, float* m_out,
                                     float* vo, void* lp, zero_dev_scalars* sc, void* ws, void* stream)
{
    ZK_CALL_RANGE();
    return fused_step(p, hp, ranks, mi, m_in, vi, mo, m_out, vo, lp, sc, ws, stream, false);
}

ZERO_API zero_status zero_step_fused_offload(const zero_plan* p, const zero_hparams* hp, const void* const* ranks,
                                             const float* mi, const float* m_in, const float* vi, float* mo,
                                             float* m_out, float* vo, void* lp, zero_dev_scalars* sc, void* ws,
                                             void* stream)
{
    ZK_CALL_RANGE();
    const void* ptrs[] = {mi, m_in, vi, mo, m_out, vo};
    for (const void* q : ptrs)
        if (!host_mapped(q)) return ZERO_ERR_INVALID_ARG;
    return fused_step(p, hp, ranks, mi, m_in, vi, mo, m_out, vo, lp, sc, ws, stream, true);
}

ZERO_API zero_status zero_accumulate_grads(const zero_plan* p, const void* const* ranks, const float* acc_in,
                                           float* acc_out, zero_dev_scalars* sc, void* stream)
{
    ZK_CALL_RANGE();
    if (p == nullptr) return ZERO_ERR_INVALID_ARG;
    zero_status s;
    if ((s = check_ranks(p, ranks)) != ZERO_OK) return s;
    if ((s = check_dev(acc_out)) != ZERO_OK) return s;
    if (acc_in != nullptr && !aligned(acc_in, 16)) return ZERO_ERR_MISALIGNED;
    if (acc_in != nullptr && acc_in != acc_out) {
        const uintptr_t i0 = reinterpret_cast<uintptr_t>(acc_in), o0 = reinterpret_cast<uintptr_t>(acc_out);
        const uintptr_t n = sizeof(float) * static_cast<uintptr_t>(p->psi);
        if (i0 < o0 + n && o0 < i0 + n) return ZERO_ERR_INVALID_ARG;
    }
    if (sc != nullptr && !aligned(sc, 256)) return ZERO_ERR_MISALIGNED;
    // the undivided sum: no loss scale, no guard; sc only reports a timeout
    StreamArgs a = base_args(nullptr, sc);
    set_ranks(a, p, ranks);
    set_flat(a, 0, p->psi);
    a.out_f32[0] = acc_out;
    a.flags = zk::F_RAW;
    set_accum(a, Accum{acc_in, 1}, 0);
    return from_cuda(zk::launch_stream(zk::OP_REDUCE, p->grad_dtype, p->param_dtype, a, as_stream(stream)));
}

ZERO_API zero_status zero_step_fused_accum(const zero_plan* p, const zero_hparams* hp, const void* const* ranks,
                                           const float* acc, int micro_batches, const float* mi, const float* m_in,
                                           const float* vi, float* mo, float* m_out, float* vo, void* lp,
                                           zero_dev_scalars* sc, void* ws, void* stream)
{
    ZK_CALL_RANGE();
    if (micro_batches < 1 || micro_batches > ZERO_MAX_MICRO_BATCHES) return ZERO_ERR_INVALID_ARG;
    if ((acc == nullptr) != (micro_batches == 1)) return ZERO_ERR_INVALID_ARG;
    if (acc != nullptr && !aligned(acc, 16)) return ZERO_ERR_MISALIGNED;
    return fused_step(p, hp, ranks, mi, m_in, vi, mo, m_out, vo, lp, sc, ws, stream, false, Accum{acc, micro_batches});
}

ZERO_API zero_status zero_quant_gather(const zero_plan* p, const void* shards, int block, signed char* codes,
                                       float* scales, void* gathered, void* stream)
{
    ZK_CALL_RANGE();
    if (p == nullptr) return ZERO_ERR_INVALID_ARG;
    if (block < 32 || block > 65536 || block % 32 != 0) return ZERO_ERR_INVALID_ARG;
    if (p->param_dtype != ZERO_BF16) return ZERO_ERR_UNSUPPORTED;
    zero_status s;
    if ((s = check_dev(shards)) != ZERO_OK) return s;
    if ((s = check_dev(codes)) != ZERO_OK) return s;
    if ((s = check_dev(scales)) != ZERO_OK) return s;
    if ((s = check_dev(gathered)) != ZERO_OK) return s;
    return from_cuda(zk::launch_quant_gather(shards, p->n_d, p->shard, p->psi, block, codes, scales, gathered,
                                             nullptr, as_stream(stream)));
}

ZERO_API zero_status zero_step_fused_qgather(const zero_plan* p, const zero_hparams* hp, const void* const* ranks,
                                             const float* mi, const float* m_in, const float* vi, float* mo,
                                             float* m_out, float* vo, int block, signed char* codes, float* scales,
                                             void* gathered, zero_dev_scalars* sc, void* ws, void* stream)
{
    ZK_CALL_RANGE();
    if (p == nullptr) return ZERO_ERR_INVALID_ARG;
    zero_status s;
    if ((s = check_hparams(hp)) != ZERO_OK) return s;
    if (block != zk::kQuantBlock) return ZERO_ERR_UNSUPPORTED;
    if (p->param_dtype != ZERO_BF16) return ZERO_ERR_UNSUPPORTED;
    const bool clip = hp->max_norm > 0.0f;
    const bool ls = hp->loss_scaling != 0;
    // loss scaling takes the guarded schedule, which leaves a skipped step's
    // state where it is: in place only
    if (ls && mo != mi) return ZERO_ERR_UNSUPPORTED;
    if ((s = check_ranks(p, ranks)) != ZERO_OK) return s;
    if ((s = check_dev(sc, 256)) != ZERO_OK) return s;
    if ((s = check_state(p, mi, m_in, vi, mo, m_out, vo)) != ZERO_OK) return s;
    if ((s = check_dev(codes)) != ZERO_OK) return s;
    if ((s = check_dev(scales)) != ZERO_OK) return s;
    if ((s = check_dev(gathered)) != ZERO_OK) return s;
    if ((clip || ls) && (s = check_dev(ws, 256)) != ZERO_OK) return s;
    const cudaStream_t st = as_stream(stream);
    int flags = zk::F_QUANT | zk::F_EPILOGUE;
    int n = 0;
    if (clip && clip_materialises(p)) {
        // the reduce pass writes the fp32 reduced gradient (and the norm
        // partials, and under loss scaling the non-finite flag); the Adam pass
        // with the int8 gather reads it instead of the ranks
        float* g = ghat_of(ws);
        if ((s = run_reduce(p, hp, ranks, g, true, ws, sc, st, &n)) != ZERO_OK) return s;
        return run_qadam(p, hp, g, mi, m_in, vi, mo, m_out, vo, codes, scales, gathered,
                         flags | zk::F_CLIP | zk::F_FINALIZE | (ls ? zk::F_GUARD : 0), sc, st, ws, n);
    }
    if (clip || ls) {
        // a read-only reduce pass first: the squared-norm partials (clipping)
        // and the non-finite flag (loss scaling); the update pass re-reads the
        // rank gradients, finishes the norm in its prologue and writes nothing
        // when the flag is set
        if ((s = run_reduce(p, hp, ranks, nullptr, clip, ws, sc, st, &n)) != ZERO_OK) return s;
        if (clip) flags |= zk::F_CLIP | zk::F_FINALIZE;
        if (ls) flags |= zk::F_GUARD | zk::F_LSCALE;
    }
    StreamArgs a = base_args(hp, sc);
    if (flags & zk::F_FINALIZE) set_finalize(a, ws, n);
    set_ranks(a, p, ranks);
    // one tile per quantization block, blocks starting at each shard's first element
    a.base = 0;
    a.seg_stride = p->shard;
    a.seg_len = p->shard;
    a.limit = p->psi;
    a.n_seg = p->n_d;
    a.tiles_per_seg = tiles_of(p->shard);
    a.q_blocks_per_shard = (p->shard + zk::kQuantBlock - 1) / zk::kQuantBlock;
    a.tma_ok = (p->shard % 8) == 0 ? 1 : 0;
    a.n_side = 3;
    a.n_side_tma = 3;
    a.side[0] = mi;
    a.side[1] = m_in;
    a.side[2] = vi;
    a.out_f32[0] = mo;
    a.out_f32[1] = m_out;
    a.out_f32[2] = vo;
    a.q_codes = codes;
    a.q_scales = scales;
    a.q_gathered = gathered;
    a.flags = flags;
    return from_cuda(zk::launch_stream(zk::OP_QFUSED, p->grad_dtype, p->param_dtype, a, st));
}

ZERO_API zero_status zero_quantize_grads(const zero_plan* p, const void* const* ranks, int block,
                                         signed char* const* codes, float* scales, zero_dev_scalars* sc,
                                         void* stream)
{
    ZK_CALL_RANGE();
    if (p == nullptr || codes == nullptr) return ZERO_ERR_INVALID_ARG;
    if (block < 32 || block > 65536 || block % 32 != 0) return ZERO_ERR_INVALID_ARG;
    if (p->grad_dtype != ZERO_BF16) return ZERO_ERR_UNSUPPORTED;
    zero_status s;
    if ((s = check_ranks(p, ranks)) != ZERO_OK) return s;
    if ((s = check_ranks(p, reinterpret_cast<const void* const*>(codes))) != ZERO_OK) return s;
    if ((s = check_dev(scales)) != ZERO_OK) return s;
    if (sc != nullptr && !aligned(sc, 256)) return ZERO_ERR_MISALIGNED;
    return from_cuda(
        zk::launch_quantize_grads(ranks, p->n_d, p->shard, p->psi, block, codes, scales, sc, as_stream(stream)));
}

ZERO_API zero_status zero_step_fused_qgz(const zero_plan* p, const zero_hparams* hp, const signed char* const* codes,
                                         const float* scales, int block, const float* mi, const float* m_in,
                                         const float* vi, float* mo, float* m_out, float* vo, void* lp,
                                         zero_dev_scalars* sc, void* ws, void* stream)
{
    ZK_CALL_RANGE();
    if (p == nullptr) return ZERO_ERR_INVALID_ARG;
    zero_status s;
    if ((s = check_hparams(hp)) != ZERO_OK) return s;
    if (block != zk::kQuantBlock) return ZERO_ERR_UNSUPPORTED;
    if (hp->loss_scaling) return ZERO_ERR_UNSUPPORTED;
    if ((s = check_ranks(p, reinterpret_cast<const void* const*>(codes))) != ZERO_OK) return s;
    if ((s = check_dev(scales)) != ZERO_OK) return s;
    if ((s = check_dev(sc, 256)) != ZERO_OK) return s;
    if ((s = check_state(p, mi, m_in, vi, mo, m_out, vo)) != ZERO_OK) return s;
    if (lp != nullptr && !aligned(lp, 16)) return ZERO_ERR_MISALIGNED;
    const bool clip = hp->max_norm > 0.0f;
    if (clip && (s = check_dev(ws, 256)) != ZERO_OK) return s;
    const cudaStream_t st = as_stream(stream);
    if (!clip) return run_fused_q8(p, hp, codes, scales, mi, m_in, vi, mo, m_out, vo, lp, zk::F_EPILOGUE, sc, st);
    // clipped: the schedule of zero_step_fused, its reduce pass over the codes
    int n = 0;
    if (clip_materialises(p)) {
        float* g = ghat_of(ws);
        if ((s = run_reduce_q8(p, hp, codes, scales, g, ws, sc, st, &n)) != ZERO_OK) return s;
        return run_adam(p, hp, g, mi, m_in, vi, mo, m_out, vo, lp,
                        zk::F_CLIP | zk::F_FINALIZE | zk::F_EPILOGUE | zk::F_REVERSE, sc, st, ws, n);
    }
    if ((s = run_reduce_q8(p, hp, codes, scales, nullptr, ws, sc, st, &n)) != ZERO_OK) return s;
    return run_fused_q8(p, hp, codes, scales, mi, m_in, vi, mo, m_out, vo, lp,
                        zk::F_CLIP | zk::F_FINALIZE | zk::F_EPILOGUE, sc, st, ws, n);
}

ZERO_API zero_status zero_step_fused_qgz_qgather(const zero_plan* p, const zero_hparams* hp,
                                                 const signed char* const* codes, const float* scales, int block,
                                                 const float* mi, const float* m_in, const float* vi, float* mo,
                                                 float* m_out, float* vo, signed char* codes_out, float* scales_out,
                                                 void* gathered, zero_dev_scalars* sc, void* ws, void* stream)
{
    ZK_CALL_RANGE();
    if (p == nullptr) return ZERO_ERR_INVALID_ARG;
    zero_status s;
    if ((s = check_hparams(hp)) != ZERO_OK) return s;
    if (block != zk::kQuantBlock) return ZERO_ERR_UNSUPPORTED;
    if (hp->loss_scaling || p->param_dtype != ZERO_BF16) return ZERO_ERR_UNSUPPORTED;
    if ((s = check_ranks(p, reinterpret_cast<const void* const*>(codes))) != ZERO_OK) return s;
    if ((s = check_dev(scales)) != ZERO_OK) return s;
    if ((s = check_dev(sc, 256)) != ZERO_OK) return s;
    if ((s = check_state(p, mi, m_in, vi, mo, m_out, vo)) != ZERO_OK) return s;
    if ((s = check_dev(codes_out)) != ZERO_OK) return s;
    if ((s = check_dev(scales_out)) != ZERO_OK) return s;
    if ((s = check_dev(gathered)) != ZERO_OK) return s;
    const bool clip = hp->max_norm > 0.0f;
    if (clip && (s = check_dev(ws, 256)) != ZERO_OK) return s;
    const cudaStream_t st = as_stream(stream);
    int flags = zk::F_QUANT | zk::F_EPILOGUE;
    int n = 0;
    if (clip && clip_materialises(p)) {
        // the reduce pass over the codes writes the fp32 reduced gradient; the
        // Adam pass with the int8 gather reads it instead of decoding again
        float* g = ghat_of(ws);
        if ((s = run_reduce_q8(p, hp, codes, scales, g, ws, sc, st, &n)) != ZERO_OK) return s;
        return run_qadam(p, hp, g, mi, m_in, vi, mo, m_out, vo, codes_out, scales_out, gathered,
                         flags | zk::F_CLIP | zk::F_FINALIZE, sc, st, ws, n);
    }
    if (clip) {
        // a read-only reduce pass over the codes; the update pass re-reads them
        if ((s = run_reduce_q8(p, hp, codes, scales, nullptr, ws, sc, st, &n)) != ZERO_OK) return s;
        flags |= zk::F_CLIP | zk::F_FINALIZE;
    }
    StreamArgs a = base_args(hp, sc);
    if (clip) set_finalize(a, ws, n);
    set_q8_ranks(a, p, codes, scales);
    a.n_side = 3;
    // N_d >= 16 int8 ranks: the state read directly, as in run_fused_q8 (both
    // ZeRO++ exchanges at N_d = 64: 4.18 -> 3.69 ms, 87% -> 99%; at N_d = 2
    // direct loads measured 22% slower)
    a.n_side_tma = p->n_d >= 2 * zk::kGroupRanks ? 0 : 3;
    a.side[0] = mi;
    a.side[1] = m_in;
    a.side[2] = vi;
    a.out_f32[0] = mo;
    a.out_f32[1] = m_out;
    a.out_f32[2] = vo;
    a.q_codes = codes_out;
    a.q_scales = scales_out;
    a.q_gathered = gathered;
    a.flags = flags;
    return from_cuda(zk::launch_stream(zk::OP_QFUSED, zk::kGradQ8, p->param_dtype, a, st));
}

ZERO_API zero_status zero_debug_wait_timeout(zero_dev_scalars* sc, long long timeout_ns, void* stream)
{
    ZK_CALL_RANGE();
    const zero_status s = check_dev(sc, 256);
    if (s != ZERO_OK) return s;
    if (timeout_ns < 1 || timeout_ns > 10000000000LL) return ZERO_ERR_INVALID_ARG;
    return from_cuda(zk::launch_debug_wait(sc, static_cast<unsigned long long>(timeout_ns), as_stream(stream)));
}

ZERO_API zero_status zero_debug_stream_timeout(int kernel, void* scratch, zero_dev_scalars* sc, long long timeout_ns,
                                               void* stream)
{
    ZK_CALL_RANGE();
    zero_status s;
    if ((s = check_dev(scratch)) != ZERO_OK) return s;
    if ((s = check_dev(sc, 256)) != ZERO_OK) return s;
    if (timeout_ns < 1 || timeout_ns > 10000000000LL) return ZERO_ERR_INVALID_ARG;
    unsigned char* buf = static_cast<unsigned char*>(scratch);
    if (kernel == 1) {
        // one 8192-element shard gathered from the first 16 KB into the next 16 KB
        const void* shards[1] = {buf};
        return from_cuda(zk::launch_all_gather(shards, 1, 8192, 8192, buf + 16384, sc, as_stream(stream), true));
    }
    if (kernel == 2) {
        // one rank, one 2048-element block: gradient in the first 4 KB, codes
        // in the next 2 KB, the scale row (4 floats) after them
        const void* ranks[1] = {buf};
        signed char* codes[1] = {reinterpret_cast<signed char*>(buf + 4096)};
        return from_cuda(zk::launch_quantize_grads(ranks, 1, 2048, 2048, zk::kQuantBlock, codes,
                                                   reinterpret_cast<float*>(buf + 8192), sc, as_stream(stream), true));
    }
    if (kernel == 3) {
        // one 2048-element shard: bf16 values in the first 4 KB, codes in the
        // next 2 KB, dequantized values at 8 KB, the scale at 12 KB
        return from_cuda(zk::launch_quant_gather(buf, 1, 2048, 2048, zk::kQuantBlock,
                                                 reinterpret_cast<signed char*>(buf + 4096),
                                                 reinterpret_cast<float*>(buf + 12288), buf + 8192, sc,
                                                 as_stream(stream), true));
    }
    if (kernel != 0) return ZERO_ERR_INVALID_ARG;
    // one full tile of one bf16 rank: the consumers wait for a stage the
    // producer never fills
    StreamArgs a = base_args(nullptr, sc);
    a.n_ranks = 1;
    a.rank[0] = scratch;
    set_flat(a, 0, zk::kTile);
    a.flags = zk::F_DEBUG_STARVE;
    a.timeout_ns = static_cast<unsigned long long>(timeout_ns);
    return from_cuda(zk::launch_stream(zk::OP_REDUCE, ZERO_BF16, ZERO_BF16, a, as_stream(stream)));
}

namespace {

// Events of one zero_step_layers call (created per call, released at its end:
// an event destroyed while work it waits on is pending is released when that
// work completes).
struct EventSet {
    cudaEvent_t* ev = nullptr;
    int n = 0;
    explicit EventSet(int count)
    {
        ev = new (std::nothrow) cudaEvent_t[count];
        if (ev == nullptr) return;
        for (; n < count; ++n)
            if (cudaEventCreateWithFlags(&ev[n], cudaEventDisableTiming) != cudaSuccess) break;
    }
    bool ok(int count) const { return ev != nullptr && n == count; }
    ~EventSet()
    {
        for (int i = 0; i < n; ++i) cudaEventDestroy(ev[i]);
        delete[] ev;
    }
    EventSet(const EventSet&) = delete;
    EventSet& operator=(const EventSet&) = delete;
};

// Workspace of the layer loop: per layer room for the partial sums of its
// reduce pass (written one after another, then finished once), then, when the
// reduced gradient goes through HBM (clipping with n_d > 4), each layer's fp32
// reduced gradient at 256-byte aligned offsets.
size_t layers_ws_bytes(const zero_hparams* hp, int n_layers, const zero_layer* layers)
{
    if (hp == nullptr || layers == nullptr || n_layers < 1) return 0;
    size_t bytes = kPartialBytes * static_cast<size_t>(n_layers);
    if (hp->max_norm > 0.0f && layers[0].plan != nullptr && clip_materialises(layers[0].plan))
        for (int l = 0; l < n_layers; ++l)
            if (layers[l].plan != nullptr)
                bytes += (sizeof(float) * static_cast<size_t>(layers[l].plan->padded) + 255) / 256 * 256;
    return bytes;
}

}  // namespace

ZERO_API size_t zero_layers_workspace_bytes(const zero_hparams* hp, int n_layers, const zero_layer* layers)
{
    return layers_ws_bytes(hp, n_layers, layers);
}

ZERO_API zero_status zero_step_layers(const zero_hparams* hp, int n_layers, const zero_layer* layers,
                                      int micro_batches, int gathers, int n_gathered, void* const* gathered,
                                      signed char* const* gathered_codes, float* const* gathered_scales,
                                      zero_dev_scalars* sc, void* ws, void* stream, void* gather_stream)
{
    ZK_CALL_RANGE();
    zero_status s;
    if ((s = check_hparams(hp)) != ZERO_OK) return s;
    if (layers == nullptr || n_layers < 1 || n_layers > ZERO_MAX_LAYERS) return ZERO_ERR_INVALID_ARG;
    if (micro_batches < 1 || micro_batches > ZERO_MAX_MICRO_BATCHES) return ZERO_ERR_INVALID_ARG;
    if (gathers < 1 || gathers > 2) return ZERO_ERR_INVALID_ARG;
    if (gathered == nullptr || n_gathered < 1 || n_gathered > n_layers) return ZERO_ERR_INVALID_ARG;
    for (int k = 0; k < n_gathered; ++k)
        if ((s = check_dev(gathered[k])) != ZERO_OK) return s;
    // quantized gathers (ZeRO++ qwZ): codes and scales for every gathered buffer, or none
    const bool qwz = gathered_codes != nullptr;
    if (qwz != (gathered_scales != nullptr)) return ZERO_ERR_INVALID_ARG;
    if (qwz) {
        for (int k = 0; k < n_gathered; ++k) {
            if ((s = check_dev(gathered_codes[k])) != ZERO_OK) return s;
            if ((s = check_dev(gathered_scales[k])) != ZERO_OK) return s;
        }
    }
    if ((s = check_dev(sc, 256)) != ZERO_OK) return s;
    const bool clip = hp->max_norm > 0.0f;
    const bool ls = hp->loss_scaling != 0;
    if ((clip || ls) && (s = check_dev(ws, 256)) != ZERO_OK) return s;
    const zero_plan* p0 = layers[0].plan;
    for (int l = 0; l < n_layers; ++l) {
        const zero_layer& L = layers[l];
        const zero_plan* p = L.plan;
        if (p == nullptr || p->stage != 3) return ZERO_ERR_INVALID_ARG;
        if (p->n_d != p0->n_d || p->grad_dtype != p0->grad_dtype || p->param_dtype != p0->param_dtype)
            return ZERO_ERR_INVALID_ARG;
        if (qwz && p->param_dtype != ZERO_BF16) return ZERO_ERR_UNSUPPORTED;
        if ((s = check_ranks(p, L.rank_grads)) != ZERO_OK) return s;
        if ((s = check_state(p, L.master, L.m, L.v, L.master, L.m, L.v)) != ZERO_OK) return s;
        if ((s = check_dev(L.shards_lp)) != ZERO_OK) return s;
        if ((L.acc == nullptr) != (micro_batches == 1)) return ZERO_ERR_INVALID_ARG;
        if (L.acc != nullptr && !aligned(L.acc, 16)) return ZERO_ERR_MISALIGNED;
        if (L.state_on_host != 0 && L.state_on_host != 1) return ZERO_ERR_INVALID_ARG;
        if (L.state_on_host && !(host_mapped(L.master) && host_mapped(L.m) && host_mapped(L.v)))
            return ZERO_ERR_INVALID_ARG;
    }
    const cudaStream_t st = as_stream(stream);
    // a second stream needs a second gathered buffer: with one, every gather
    // waits for the step before it, which leaves nothing to overlap
    const cudaStream_t gs = gather_stream != nullptr && n_gathered >= 2 ? as_stream(gather_stream) : st;
    const bool two = gs != st;
    // events: [0] the call's start on `stream`, [1 + l] layer l gathered,
    // [1 + n + l] layer l stepped, [1 + 2n] the gather stream's end
    const int n_ev = two ? 2 * n_layers + 2 : 0;
    EventSet ev(n_ev);
    if (two && !ev.ok(n_ev)) return ZERO_ERR_CUDA;
    const int n_d = p0->n_d;
    const void* shard_ptr[ZERO_MAX_RANKS];
    const bool materialise = clip && clip_materialises(p0);
    auto acc_of = [&](const zero_layer& L) { return Accum{L.acc, micro_batches}; };
    // the workspace: partial sums of every layer's reduce pass, one after
    // another, then the layers' reduced gradients
    double* partials = partials_of(ws);
    // layer l's reduced gradient: walked layer by layer in both loops below
    // (each region 256-byte aligned), so no layer is looked up by a search
    const size_t ghat_base = kPartialBytes * static_cast<size_t>(n_layers);
    auto ghat_size = [&](int l) {
        return (sizeof(float) * static_cast<size_t>(layers[l].plan->padded) + 255) / 256 * 256;
    };
    auto ghat_ptr = [&](size_t off) { return reinterpret_cast<float*>(static_cast<char*>(ws) + ghat_base + off); };

    // The global checks span every layer: with clipping or loss scaling a
    // reduce pass over each layer first (norm partials, the non-finite flag;
    // the reduced gradient too when it goes through HBM), the norm finished
    // once, then the updates, each applying the one coefficient (and all
    // skipped together when a value was not finite).
    if (clip || ls) {
        int n_part = 0;
        size_t g_off = 0;
        for (int l = 0; l < n_layers; ++l) {
            const zero_layer& L = layers[l];
            if (L.grads_ready != nullptr) ZK_TRY(cudaStreamWaitEvent(st, static_cast<cudaEvent_t>(L.grads_ready), 0));
            int grid = 0;
            if ((s = run_reduce(L.plan, hp, L.rank_grads, materialise ? ghat_ptr(g_off) : nullptr, clip,
                                partials + n_part, sc, st, &grid, acc_of(L))) != ZERO_OK)
                return s;
            if (clip) n_part += grid;
            g_off += ghat_size(l);
        }
        if (clip) ZK_TRY(zk::launch_finalize_sqnorm(partials, n_part, *hp, sc, st));
    }

    // gather(l): layer l's 16-bit shards into gathered[l % n_gathered], once
    // or twice (forward and backward); it waits for the step that last used
    // that buffer (layer l - n_gathered) -- its own shards were last written
    // before this call, which the gather stream waits for at the start
    auto gather = [&](int l) -> zero_status {
        const zero_layer& L = layers[l];
        const zero_plan* p = L.plan;
        if (two && l >= n_gathered) ZK_TRY(cudaStreamWaitEvent(gs, ev.ev[1 + n_layers + l - n_gathered], 0));
        const size_t eb = 2;   // 16-bit parameters
        for (int r = 0; r < n_d; ++r)
            shard_ptr[r] = static_cast<const unsigned char*>(L.shards_lp) + eb * static_cast<size_t>(r) * p->shard;
        const int k = l % n_gathered;
        for (int g = 0; g < gathers; ++g) {
            if (qwz)
                ZK_TRY(zk::launch_quant_gather(L.shards_lp, n_d, p->shard, p->psi, zk::kQuantBlock,
                                               gathered_codes[k], gathered_scales[k], gathered[k], sc, gs));
            else
                ZK_TRY(zk::launch_all_gather(shard_ptr, n_d, p->shard, p->psi, gathered[k], sc, gs));
        }
        if (two) ZK_TRY(cudaEventRecord(ev.ev[1 + l], gs));
        return ZERO_OK;
    };

    if (two) {
        ZK_TRY(cudaEventRecord(ev.ev[0], st));
        ZK_TRY(cudaStreamWaitEvent(gs, ev.ev[0], 0));
    }
    if ((s = gather(0)) != ZERO_OK) return s;
    const int flags = (clip ? zk::F_CLIP : 0) | (ls ? (zk::F_GUARD | zk::F_LSCALE) : 0);
    size_t g_off = 0;
    for (int l = 0; l < n_layers; ++l) {
        // the next layer's gather is issued before this layer's step, so that
        // with two streams it runs while the step does
        if (two && l + 1 < n_layers && (s = gather(l + 1)) != ZERO_OK) return s;
        if (two) ZK_TRY(cudaStreamWaitEvent(st, ev.ev[1 + l], 0));
        const zero_layer& L = layers[l];
        if (!(clip || ls) && L.grads_ready != nullptr)
            ZK_TRY(cudaStreamWaitEvent(st, static_cast<cudaEvent_t>(L.grads_ready), 0));
        // no scalar commit per layer: every layer's Adam takes this step's t
        const bool host = L.state_on_host != 0;
        float* ghat = ghat_ptr(g_off);
        g_off += ghat_size(l);
        if (materialise)
            s = run_adam(L.plan, hp, ghat, L.master, L.m, L.v, L.master, L.m, L.v, L.shards_lp,
                         flags & ~zk::F_LSCALE, sc, st, nullptr, 0, host);
        else
            s = run_fused(L.plan, hp, L.rank_grads, L.master, L.m, L.v, L.master, L.m, L.v, L.shards_lp, flags, sc,
                          st, nullptr, 0, host, acc_of(L));
        if (s != ZERO_OK) return s;
        if (two) ZK_TRY(cudaEventRecord(ev.ev[1 + n_layers + l], st));
        if (L.stepped != nullptr) ZK_TRY(cudaEventRecord(static_cast<cudaEvent_t>(L.stepped), st));
        if (!two && l + 1 < n_layers && (s = gather(l + 1)) != ZERO_OK) return s;
    }
    if (two) {
        ZK_TRY(cudaEventRecord(ev.ev[1 + 2 * n_layers], gs));
        ZK_TRY(cudaStreamWaitEvent(st, ev.ev[1 + 2 * n_layers], 0));
    }
    // the step scalars advance once for the whole stack (or, after a
    // non-finite value, the step is skipped and the scale halves)
    return from_cuda(zk::launch_epilogue(*hp, sc, st));
}

ZERO_API unsigned long long zero_launch_count(void) { return zk::launch_count(); }

}  // extern "C"
