// zk_aux.cu -- the smaller kernels of the ZeRO-DP step.
//
//   k_all_gather     shard r's valid elements -> gathered[r*S ...] through a
//                    ring of shared-memory stages filled and drained by 1-D
//                    bulk copies (DP-notes "ZeRO-1": gather the updated
//                    partitions; itwiki: ZeRO-3 gathers each layer before use)
//   k_quant_gather   block-int8 quantize + dequantize of the bf16 shards
//                    (itwiki "후속 기법", ZeRO++ qwZ), per-warp bulk-copy slots
//   k_quantize_ranks every rank's gradient through the block quantizer in one
//                    launch (ZeRO++ qgZ sender), per-warp bulk-copy slots
//   k_sqnorm_f32     per-CTA partial sums of g^2 of an fp32 array
//   k_finalize       fixed-order fp64 sum of the partials, clip coefficient
//   k_epilogue       commits the step scalars (t, beta powers, loss scale)
//   k_repair         restores a speculative step that turned out to overflow
//   k_scalars_init, k_debug_wait
#include <cstring>

#include "zk_common.cuh"
#include "zk_launch.h"

namespace zk {

namespace {

unsigned long long g_launches = 0;

int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace

void count_launch() { __atomic_add_fetch(&g_launches, 1ull, __ATOMIC_RELAXED); }
unsigned long long launch_count() { return __atomic_load_n(&g_launches, __ATOMIC_RELAXED); }

// ------------------------------------------------------------------ scalars
__global__ void k_scalars_init(zero_dev_scalars* sc, float loss_scale)
{
    zero_dev_scalars s = {};
    s.t = 0;
    s.beta1_pow = 1.0;
    s.beta2_pow = 1.0;
    s.sqnorm = 0.0;
    s.loss_scale = loss_scale;
    s.clip_coef = 1.0f;
    *sc = s;
}

cudaError_t launch_scalars_init(zero_dev_scalars* sc, float loss_scale, cudaStream_t st)
{
    count_launch();
    k_scalars_init<<<1, 1, 0, st>>>(sc, loss_scale);
    return cudaGetLastError();
}

// Commits (or skips) the step: commit_scalars in zk_common.cuh.
__global__ void k_epilogue(zero_hparams hp, zero_dev_scalars* sc) { commit_scalars(hp, sc); }

cudaError_t launch_epilogue(const zero_hparams& hp, zero_dev_scalars* sc, cudaStream_t st)
{
    count_launch();
    k_epilogue<<<1, 1, 0, st>>>(hp, sc);
    return cudaGetLastError();
}

// --------------------------------------------------------------- squared norm
// Fixed-order fp64 sum of the per-CTA partials by one warp (lane l takes
// partials l, l+32, ... in order; then a butterfly that gives every lane the
// same bits), then norm and coefficient: coef = max_norm / (norm + 1e-6),
// applied when below one.
__global__ void k_finalize(const double* partials, int n, zero_hparams hp, zero_dev_scalars* sc)
{
    double x = 0.0;
    for (int i = threadIdx.x; i < n; i += 32) x = __dadd_rn(x, partials[i]);
    x = warp_sum_f64(x);
    if (threadIdx.x == 0) {
        sc->sqnorm = x;
        sc->clip_coef = clip_coefficient(hp.max_norm, x);
    }
}

cudaError_t launch_finalize_sqnorm(const double* partials, int n, const zero_hparams& hp,
                                   zero_dev_scalars* sc, cudaStream_t st)
{
    count_launch();
    k_finalize<<<1, 32, 0, st>>>(partials, n, hp, sc);
    return cudaGetLastError();
}

__global__ void __launch_bounds__(256) k_sqnorm_f32(const float* __restrict__ g, long long n, double* partials)
{
    float hi = 0.0f, lo = 0.0f;
    const long long n4 = n / 4;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
        const float4 f = reinterpret_cast<const float4*>(g)[i];
        sq_accumulate(f.x, hi, lo);
        sq_accumulate(f.y, hi, lo);
        sq_accumulate(f.z, hi, lo);
        sq_accumulate(f.w, hi, lo);
    }
    if (blockIdx.x == 0 && threadIdx.x < n - n4 * 4) sq_accumulate(g[n4 * 4 + threadIdx.x], hi, lo);
    __shared__ double red[8];
    double part = warp_sum_f64(__dadd_rn(static_cast<double>(hi), static_cast<double>(lo)));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = part;
    __syncthreads();
    if (threadIdx.x == 0) {
        double tot = 0.0;
        for (int w = 0; w < 8; ++w) tot = __dadd_rn(tot, red[w]);
        partials[blockIdx.x] = tot;
    }
}

cudaError_t launch_sqnorm_f32(const float* g, long long n, double* partials, int* n_partials, cudaStream_t st)
{
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    long long blocks = (n / 4 + 255) / 256;
    if (blocks > 4LL * sms) blocks = 4LL * sms;
    if (blocks > kMaxPartials) blocks = kMaxPartials;
    if (blocks < 1) blocks = 1;
    *n_partials = static_cast<int>(blocks);
    count_launch();
    k_sqnorm_f32<<<static_cast<unsigned>(blocks), 256, 0, st>>>(g, n, partials);
    return cudaGetLastError();
}

// ----------------------------------------------------------------- repair
// Speculative loss-scaled step that met a non-finite gradient: the out state
// gets the in state back and the 16-bit parameters are re-cast from it.
template <int PT>
__global__ void k_repair(const float* __restrict__ mi, const float* __restrict__ m_in,
                         const float* __restrict__ v_in, float* mo, float* m_out, float* v_out,
                         uint16_t* lp, long long psi, const zero_dev_scalars* sc)
{
    if (sc->nonfinite == 0) return;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long j = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; j < psi; j += stride) {
        const float p = mi[j];
        if (mo != mi) {
            mo[j] = p;
            m_out[j] = m_in[j];
            v_out[j] = v_in[j];
        }
        if (lp != nullptr) lp[j] = Lp<PT>::narrow(p);
    }
}

cudaError_t launch_repair(const float* master_in, const float* m_in, const float* v_in, float* master_out,
                          float* m_out, float* v_out, void* lp_out, int param_dtype, long long psi, zero_dev_scalars* sc,
                          cudaStream_t st)
{
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    long long blocks = (psi + 255) / 256;
    if (blocks > 8LL * sms) blocks = 8LL * sms;
    if (blocks < 1) blocks = 1;
    uint16_t* lp = static_cast<uint16_t*>(lp_out);
    count_launch();
    if (param_dtype == ZERO_BF16)
        k_repair<ZERO_BF16><<<static_cast<unsigned>(blocks), 256, 0, st>>>(master_in, m_in, v_in, master_out, m_out, v_out, lp, psi, sc);
    else
        k_repair<ZERO_FP16><<<static_cast<unsigned>(blocks), 256, 0, st>>>(master_in, m_in, v_in, master_out, m_out, v_out, lp, psi, sc);
    return cudaGetLastError();
}

// --------------------------------------------------------------- all-gather
constexpr int kAgTile = 8192;    // 16-bit elements per bulk copy (16 KB)
constexpr int kAgStages = 8;
constexpr int kAgThreads = 256;

struct AgArgs {
    const void* shard[ZERO_MAX_RANKS];
    void* gathered;
    long long shard_len;          // S
    long long psi;
    long long tiles_per_shard;    // ceil(S / kAgTile)
    int n_d;
    int tma_ok;                   // S % 8 == 0 (every tile 16-byte aligned at both ends)
    int starve;                   // issue no copy: every wait runs out (tests the timeout path)
    unsigned long long timeout_ns;
    zero_dev_scalars* sc;
};

__device__ __forceinline__ void ag_span(const AgArgs& a, long long tile, int& r, long long& i0, int& len)
{
    r = static_cast<int>(tile / a.tiles_per_shard);
    i0 = (tile - static_cast<long long>(r) * a.tiles_per_shard) * kAgTile;
    long long valid = a.psi - static_cast<long long>(r) * a.shard_len;
    valid = valid < 0 ? 0 : (valid > a.shard_len ? a.shard_len : valid);
    const long long l = valid - i0;
    len = l <= 0 ? 0 : (l > kAgTile ? kAgTile : static_cast<int>(l));
}

__global__ void __launch_bounds__(kAgThreads) k_all_gather(const __grid_constant__ AgArgs a)
{
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    int* issued = reinterpret_cast<int*>(smem + 8 * kAgStages);
    unsigned char* ring = smem + 1024;
    const long long ntiles = a.tiles_per_shard * a.n_d;
    uint16_t* out = static_cast<uint16_t*>(a.gathered);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kAgStages; ++s) {
            mbar_init(&full[s], 1);
            issued[s] = -1;
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (threadIdx.x < 32) {
        if (threadIdx.x == 0 && a.tma_ok) {
            // one thread drives the ring: bulk load tile -> stage, bulk store stage -> gathered
            auto next_full = [&](long long t) {
                for (; t < ntiles; t += gridDim.x) {
                    int r;
                    long long i0;
                    int len;
                    ag_span(a, t, r, i0, len);
                    if (len == kAgTile) return t;
                }
                return ntiles;
            };
            auto issue_load = [&](long long t, int s, uint32_t ph) {
                if (a.starve) return;
                int r;
                long long i0;
                int len;
                ag_span(a, t, r, i0, len);
                mbar_arrive_expect_tx(&full[s], kAgTile * 2);
                bulk_load(ring + s * (kAgTile * 2), static_cast<const uint16_t*>(a.shard[r]) + i0, kAgTile * 2, &full[s]);
                issued[s] = static_cast<int>(ph);
            };
            long long load_t = next_full(blockIdx.x);
            long long k_load = 0;
            for (int s = 0; s < kAgStages && load_t < ntiles; ++s) {
                issue_load(load_t, s, 0u);
                ++k_load;
                load_t = next_full(load_t + gridDim.x);
            }
            long long k = 0;
            bool ok = true;
            for (long long t = next_full(blockIdx.x); t < ntiles; t = next_full(t + gridDim.x), ++k) {
                const int s = static_cast<int>(k % kAgStages);
                const uint32_t ph = static_cast<uint32_t>((k / kAgStages) & 1);
                if (!mbar_wait_bounded(&full[s], ph, nullptr, a.timeout_ns)) {
                    ok = false;
                    break;
                }
                int r;
                long long i0;
                int len;
                ag_span(a, t, r, i0, len);
                bulk_store(out + static_cast<long long>(r) * a.shard_len + i0, ring + s * (kAgTile * 2), kAgTile * 2);
                bulk_commit();
                if (k >= 1 && load_t < ntiles) {
                    // the store of tile k-1 has finished reading its stage: refill it
                    bulk_wait_read<1>();
                    const long long kk = k - 1 + kAgStages;
                    issue_load(load_t, static_cast<int>((k - 1) % kAgStages), static_cast<uint32_t>((kk / kAgStages) & 1));
                    ++k_load;
                    load_t = next_full(load_t + gridDim.x);
                }
            }
            bulk_wait_all<0>();
            if (!ok) {
                for (int s = 0; s < kAgStages; ++s)
                    if (issued[s] >= 0) mbar_wait_bounded(&full[s], static_cast<uint32_t>(issued[s]), nullptr, a.timeout_ns);
                if (a.sc != nullptr) atomicOr(&a.sc->status, ZERO_DEV_TIMEOUT);
            }
        }
        __syncwarp();
    } else {
        // warps 1..7: tiles the ring does not take (short, or unaligned shards)
        const int t0 = threadIdx.x - 32;
        const int nt = kAgThreads - 32;
        for (long long t = blockIdx.x; t < ntiles; t += gridDim.x) {
            int r;
            long long i0;
            int len;
            ag_span(a, t, r, i0, len);
            if (len <= 0 || (len == kAgTile && a.tma_ok)) continue;
            const uint16_t* src = static_cast<const uint16_t*>(a.shard[r]) + i0;
            uint16_t* dst = out + static_cast<long long>(r) * a.shard_len + i0;
            for (int i = t0; i < len; i += nt) dst[i] = src[i];
        }
    }
    __syncthreads();
}

cudaError_t launch_all_gather(const void* const* shards, int n_d, long long shard, long long psi,
                              void* gathered, zero_dev_scalars* sc, cudaStream_t st, bool starve)
{
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    AgArgs a = {};
    for (int r = 0; r < n_d; ++r) a.shard[r] = shards[r];
    a.gathered = gathered;
    a.shard_len = shard;
    a.psi = psi;
    a.tiles_per_shard = (shard + kAgTile - 1) / kAgTile;
    a.n_d = n_d;
    bool aligned = shard % 8 == 0 && (reinterpret_cast<uintptr_t>(gathered) & 15) == 0;
    for (int r = 0; r < n_d; ++r) aligned = aligned && (reinterpret_cast<uintptr_t>(shards[r]) & 15) == 0;
    a.tma_ok = aligned ? 1 : 0;
    a.timeout_ns = starve ? 2000000ull : kDefaultTimeoutNs;
    a.starve = starve ? 1 : 0;
    a.sc = sc;
    const long long ntiles = a.tiles_per_shard * n_d;
    if (ntiles <= 0) return cudaSuccess;
    const size_t smem = 1024 + static_cast<size_t>(kAgStages) * kAgTile * 2;
    static int attr_done[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !__atomic_load_n(&attr_done[dev], __ATOMIC_ACQUIRE)) {
        cudaError_t e = cudaFuncSetAttribute(k_all_gather, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        __atomic_store_n(&attr_done[dev], 1, __ATOMIC_RELEASE);
    }
    long long grid = ntiles < sms ? ntiles : sms;
    count_launch();
    k_all_gather<<<static_cast<unsigned>(grid), kAgThreads, smem, st>>>(a);
    return cudaGetLastError();
}

// ------------------------------------------------------- quantized gather
// The qwZ weight gather: the flat bf16 shards through the block quantizer,
// codes and dequantized bf16 at the global index, scales at [r * nbs + b].
// The same pipeline as the gradient sender below: one warp per 2048-element
// block at a time, kQgSlots shared-memory slots per warp that its lane 0
// fills with 1-D bulk copies kQgSlots blocks ahead, no block-wide barrier.
// 20 warps (96 registers: the dequantized output needs more than 24 warps
// leave).  Blocks that are not full, 16-byte aligned 2048-element blocks
// (ragged shard ends, other block sizes) are read from global memory twice
// (amax, then codes).  A wait that runs out is reported when a scalars block
// is given, and the warp then reads that block and every later one from
// global memory, so the results stay complete either way.
constexpr int kQgWarps = 20;
constexpr int kQgSlots = 2;
constexpr int kQgSlotBytes = kQuantBlock * 2;

struct QgArgs {
    const uint16_t* shards;
    signed char* codes;
    uint16_t* gathered;
    float* scales;
    zero_dev_scalars* sc;                 // may be null
    long long shard, psi, nbs, total;     // total = n_d * nbs blocks
    int block, ring_ok;                   // ring_ok: block == 2048, shard % 8 == 0, 16-byte aligned buffers
    int starve;                           // issue no copy: every wait runs out (tests the fallback)
    unsigned long long timeout_ns;
};

struct QgBlock {
    long long bi;    // block index r * nbs + b (its scale's index)
    long long j0;    // first element (global index)
    int n;           // valid elements (0: past psi)
};

__device__ __forceinline__ QgBlock qg_block(const QgArgs& a, long long bi)
{
    QgBlock k;
    k.bi = bi;
    const long long r = bi / a.nbs;
    const long long lo = (bi - r * a.nbs) * a.block;
    long long valid = a.psi - r * a.shard;
    valid = valid < 0 ? 0 : (valid > a.shard ? a.shard : valid);
    const long long hi = lo + a.block < valid ? lo + a.block : valid;
    k.j0 = r * a.shard + lo;
    k.n = hi > lo ? static_cast<int>(hi - lo) : 0;
    return k;
}

// |x| maxima of a slot's 2048 bf16 values on bf16 pairs (a max picks one of
// its inputs, so it is exact in bf16; a NaN input is passed over as fmaxf
// does), over the warp: the block's scale amax / 127
__device__ __forceinline__ float slot_scale(const uint4* src, int lane)
{
    __nv_bfloat162 am[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) am[e] = __float2bfloat162_rn(0.0f);
#pragma unroll
    for (int v = 0; v < 8; ++v) {
        const uint4 wv = src[v * 32 + lane];
        const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) am[e] = __hmax2(am[e], __habs2(*reinterpret_cast<const __nv_bfloat162*>(&ws[e])));
    }
    const __nv_bfloat162 m2 = __hmax2(__hmax2(am[0], am[1]), __hmax2(am[2], am[3]));
    const float amax = warp_max_f32(fmaxf(__low2float(m2), __high2float(m2)));
    return __fdiv_rn(amax, 127.0f);
}

__global__ void __launch_bounds__(kQgWarps * 32, 1) k_quant_gather(const __grid_constant__ QgArgs a)
{
    extern __shared__ __align__(1024) unsigned char smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem) + warp * kQgSlots;
    unsigned char* slot0 = smem + 1024 + static_cast<size_t>(warp) * kQgSlots * kQgSlotBytes;
    const long long step = static_cast<long long>(gridDim.x) * kQgWarps;
    const long long first = static_cast<long long>(blockIdx.x) * kQgWarps + warp;

    if (lane == 0) {
        for (int s = 0; s < kQgSlots; ++s) mbar_init(&bar[s], 1);
        fence_barrier_init();
    }
    __syncwarp();

    bool ring = true;       // warp-uniform: cleared when a wait runs out
    uint32_t pending = 0;   // lane 0: slots with a copy in flight
    long long ib = first;   // issue cursor, kQgSlots blocks ahead of the work cursor
    auto issue = [&](int s) {
        if (ib < a.total) {
            const QgBlock k = qg_block(a, ib);
            if (ring && a.ring_ok && k.n == kQuantBlock && lane == 0 && !a.starve) {
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(&bar[s], kQgSlotBytes);
                bulk_load(slot0 + s * kQgSlotBytes, a.shards + k.j0, kQgSlotBytes, &bar[s]);
                pending |= 1u << s;
            }
        }
        ib += step;
    };
    // a block read from global memory twice (amax, then codes)
    auto from_global = [&](const QgBlock& k) {
        const uint16_t* x = a.shards + k.j0;
        float amax = 0.0f;
        for (int i = lane; i < k.n; i += 32) amax = fmaxf(amax, fabsf(Lp<ZERO_BF16>::widen(x[i])));
        amax = warp_max_f32(amax);
        const float sc = __fdiv_rn(amax, 127.0f);
        if (lane == 0) a.scales[k.bi] = sc;
        const float inv = quant_reciprocal(sc);
        for (int i = lane; i < k.n; i += 32) {
            const float cf = quant_code_f(Lp<ZERO_BF16>::widen(x[i]), sc, inv);
            a.codes[k.j0 + i] = static_cast<signed char>(static_cast<uint8_t>(code_bits(cf)));
            a.gathered[k.j0 + i] = Lp<ZERO_BF16>::narrow(__fmul_rn(cf, sc));
        }
    };
    for (int s = 0; s < kQgSlots; ++s) issue(s);

    uint32_t phase = 0;     // per slot: parity of its next completion
    bool timed_out = false;
    int s = 0;
    for (long long bi = first; bi < a.total; bi += step, s = (s + 1 == kQgSlots) ? 0 : s + 1) {
        const QgBlock k = qg_block(a, bi);
        if (k.n <= 0) {
            if (lane == 0) a.scales[k.bi] = 0.0f;
            issue(s);
            continue;
        }
        if (ring && a.ring_ok && k.n == kQuantBlock) {
            const bool got = mbar_wait_bounded(&bar[s], (phase >> s) & 1u, nullptr, a.timeout_ns);
            if (!__all_sync(0xffffffffu, got)) {
                // the copy did not land in time: this block and the rest from global memory
                timed_out = true;
                ring = false;
                issue(s);
                from_global(k);
                continue;
            }
            phase ^= 1u << s;
            if (lane == 0) pending &= ~(1u << s);
            // the block is read from its slot twice (amax, then codes) so that a
            // lane holds 16 bytes of it at a time
            const uint4* src = reinterpret_cast<const uint4*>(slot0 + s * kQgSlotBytes);
            const float sc = slot_scale(src, lane);
            if (lane == 0) a.scales[k.bi] = sc;
            const float inv = quant_reciprocal(sc);
            uint2* dst = reinterpret_cast<uint2*>(a.codes + k.j0);
            uint4* gdst = reinterpret_cast<uint4*>(a.gathered + k.j0);
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const uint4 wv = src[v * 32 + lane];
                const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
                uint32_t packed[2], dq[4];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float xs[4] = {Lp<ZERO_BF16>::lo(ws[2 * h]), Lp<ZERO_BF16>::hi(ws[2 * h]),
                                         Lp<ZERO_BF16>::lo(ws[2 * h + 1]), Lp<ZERO_BF16>::hi(ws[2 * h + 1])};
                    float cf[4];
                    packed[h] = quant_code4(xs, sc, inv, cf);
                    dq[2 * h] = Lp<ZERO_BF16>::narrow2(__fmul_rn(cf[0], sc), __fmul_rn(cf[1], sc));
                    dq[2 * h + 1] = Lp<ZERO_BF16>::narrow2(__fmul_rn(cf[2], sc), __fmul_rn(cf[3], sc));
                }
                dst[v * 32 + lane] = make_uint2(packed[0], packed[1]);
                gdst[v * 32 + lane] = make_uint4(dq[0], dq[1], dq[2], dq[3]);
            }
            // every lane's reads of the slot are complete (their values were used): refill it
            __syncwarp();
            issue(s);
        } else {
            issue(s);
            from_global(k);
        }
    }
    if (timed_out && lane == 0) {
        // let the copies in flight land before the CTA's shared memory is released
        for (int t = 0; t < kQgSlots; ++t)
            if (pending & (1u << t)) mbar_wait_bounded(&bar[t], (phase >> t) & 1u, nullptr, a.timeout_ns);
        if (a.sc != nullptr) atomicOr(&a.sc->status, ZERO_DEV_TIMEOUT);
    }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

cudaError_t launch_quant_gather(const void* shards, int n_d, long long shard, long long psi, int block,
                                signed char* codes, float* scales, void* gathered, zero_dev_scalars* sc,
                                cudaStream_t st, bool starve)
{
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    QgArgs a;
    std::memset(&a, 0, sizeof(a));
    a.shards = static_cast<const uint16_t*>(shards);
    a.codes = codes;
    a.gathered = static_cast<uint16_t*>(gathered);
    a.scales = scales;
    a.sc = sc;
    a.shard = shard;
    a.psi = psi;
    a.block = block;
    a.nbs = (shard + block - 1) / block;
    a.total = static_cast<long long>(n_d) * a.nbs;
    a.ring_ok = (block == kQuantBlock && shard % 8 == 0 && aligned16(shards) && aligned16(codes) &&
                 aligned16(gathered)) ? 1 : 0;
    a.timeout_ns = starve ? 2000000ull : kDefaultTimeoutNs;
    a.starve = starve ? 1 : 0;
    if (a.total <= 0) return cudaSuccess;
    const size_t smem = 1024 + static_cast<size_t>(kQgWarps) * kQgSlots * kQgSlotBytes;
    static int attr_done[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (dev < 64 && !__atomic_load_n(&attr_done[dev], __ATOMIC_ACQUIRE)) {
        const cudaError_t e =
            cudaFuncSetAttribute(k_quant_gather, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        __atomic_store_n(&attr_done[dev], 1, __ATOMIC_RELEASE);
    }
    long long grid = (a.total + kQgWarps - 1) / kQgWarps;
    if (grid > sms) grid = sms;
    count_launch();
    k_quant_gather<<<static_cast<unsigned>(grid), kQgWarps * 32, smem, st>>>(a);
    return cudaGetLastError();
}

// Sender side of the quantized gradient exchange: every rank q's bf16
// gradient through the block quantizer, codes at the global index of rank
// q's code buffer, scales at [(r * nbs + b) * n_dp + q] (block b of shard r).
// All ranks in one launch.  One warp per block at a time, no block-wide
// barrier: each warp owns kQsSlots shared-memory slots of one 2048-element
// block that its lane 0 fills with 1-D bulk copies kQsSlots blocks ahead, so
// ~192 KB per SM are in flight while the warps quantize.  Blocks that are not
// full, 16-byte aligned 2048-element blocks (ragged shard ends, other block
// sizes) are read from global memory twice (amax, then codes).
constexpr int kQsWarps = 24;
constexpr int kQsSlots = 2;
constexpr int kQsSlotBytes = kQuantBlock * 2;

struct QsArgs {
    const uint16_t* rank[ZERO_MAX_RANKS];
    signed char* codes[ZERO_MAX_RANKS];
    float* scales;
    zero_dev_scalars* sc;                     // may be null: receives ZERO_DEV_TIMEOUT
    long long shard, psi, nbs, n_dp, total;   // total = n_d * n_d * nbs blocks
    int n_d, block, ring_ok;                   // ring_ok: block == 2048 and shard % 8 == 0
    int starve;                                // issue no copy: every wait runs out (tests the timeout path)
    unsigned long long timeout_ns;
};

struct QsBlock {
    int q;           // rank whose gradient it is
    long long row;   // scale row r * nbs + b
    long long j0;    // first element (global index)
    int n;           // valid elements (0: past psi)
};

// Walks one warp's blocks bi = first, first + step, ... as (q, r, b) with
// bi = (q * n_d + r) * nbs + b: divisions once, then add-and-carry.
struct QsCursor {
    int q, r, b;      // current block (nbs < 2^31: checked at launch)
    int dq, dr, db;   // step split the same way

    __device__ static __forceinline__ void split(const QsArgs& a, long long x, int& q, int& r, int& b)
    {
        const long long per_rank = static_cast<long long>(a.n_d) * a.nbs;
        const long long qq = x / per_rank;
        const long long row = x - qq * per_rank;
        const long long rr = row / a.nbs;
        q = static_cast<int>(qq);   // x < grid * warps per CTA: fits
        r = static_cast<int>(rr);
        b = static_cast<int>(row - rr * a.nbs);
    }
    __device__ __forceinline__ void start(const QsArgs& a, long long first, long long step)
    {
        split(a, first, q, r, b);
        split(a, step, dq, dr, db);
    }
    __device__ __forceinline__ void next(const QsArgs& a)
    {
        b += db;
        if (b >= a.nbs) {
            b -= a.nbs;
            ++r;
        }
        r += dr;
        if (r >= a.n_d) {
            r -= a.n_d;
            ++q;
        }
        q += dq;
    }
    __device__ __forceinline__ bool valid(const QsArgs& a) const { return q < a.n_d; }
    __device__ __forceinline__ QsBlock block(const QsArgs& a) const
    {
        QsBlock k;
        k.q = q;
        k.row = static_cast<long long>(r) * a.nbs + b;
        long long valid = a.psi - static_cast<long long>(r) * a.shard;
        valid = valid < 0 ? 0 : (valid > a.shard ? a.shard : valid);
        const long long lo = static_cast<long long>(b) * a.block;
        const long long hi = lo + a.block < valid ? lo + a.block : valid;
        k.j0 = static_cast<long long>(r) * a.shard + lo;
        k.n = hi > lo ? static_cast<int>(hi - lo) : 0;
        return k;
    }
};

__device__ __forceinline__ bool qs_ring(const QsArgs& a, const QsBlock& k) { return a.ring_ok && k.n == kQuantBlock; }

__global__ void __launch_bounds__(kQsWarps * 32, 1) k_quantize_ranks(const __grid_constant__ QsArgs a)
{
    extern __shared__ __align__(1024) unsigned char smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem) + warp * kQsSlots;
    unsigned char* slot0 = smem + 1024 + static_cast<size_t>(warp) * kQsSlots * kQsSlotBytes;
    const long long step = static_cast<long long>(gridDim.x) * kQsWarps;
    const long long first = static_cast<long long>(blockIdx.x) * kQsWarps + warp;
    const int pad = static_cast<int>(a.n_dp) - a.n_d;

    if (lane == 0) {
        for (int s = 0; s < kQsSlots; ++s) mbar_init(&bar[s], 1);
        fence_barrier_init();
    }
    __syncwarp();

    // lane 0 issues the block under the issue cursor, kQsSlots blocks ahead
    // of the work cursor, into slot s
    uint32_t pending = 0;   // lane 0: slots with a copy in flight
    QsCursor ic;
    ic.start(a, first, step);
    auto issue = [&](int s) {
        if (ic.valid(a)) {
            const QsBlock k = ic.block(a);
            if (qs_ring(a, k) && lane == 0 && !a.starve) {
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(&bar[s], kQsSlotBytes);
                bulk_load(slot0 + s * kQsSlotBytes, a.rank[k.q] + k.j0, kQsSlotBytes, &bar[s]);
                pending |= 1u << s;
            }
        }
        ic.next(a);
    };
    for (int s = 0; s < kQsSlots; ++s) issue(s);

    uint32_t phase = 0;     // per slot: parity of its next completion
    bool ok = true;
    QsCursor wc;
    wc.start(a, first, step);
    for (int s = 0; wc.valid(a); wc.next(a), s = (s + 1 == kQsSlots) ? 0 : s + 1) {
        const QsBlock k = wc.block(a);
        float* srow = a.scales + k.row * a.n_dp;
        if (k.q == a.n_d - 1 && lane >= 1 && lane <= pad) srow[a.n_d - 1 + lane] = 0.0f;   // layout padding
        if (k.n <= 0) {
            if (lane == 0) srow[k.q] = 0.0f;
            issue(s);
            continue;
        }
        if (qs_ring(a, k)) {
            const bool got = mbar_wait_bounded(&bar[s], (phase >> s) & 1u, nullptr, a.timeout_ns);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            phase ^= 1u << s;
            if (lane == 0) pending &= ~(1u << s);
            // the block is read from its slot twice (amax, then codes) so that a
            // lane holds 16 bytes of it at a time
            const uint4* src = reinterpret_cast<const uint4*>(slot0 + s * kQsSlotBytes);
            // |x| maxima on bf16 pairs (a max picks one of its inputs, so it is
            // exact in bf16; a NaN input is passed over as fmaxf does)
            __nv_bfloat162 am[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) am[e] = __float2bfloat162_rn(0.0f);
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const uint4 wv = src[v * 32 + lane];
                const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) am[e] = __hmax2(am[e], __habs2(*reinterpret_cast<const __nv_bfloat162*>(&ws[e])));
            }
            const __nv_bfloat162 m2 = __hmax2(__hmax2(am[0], am[1]), __hmax2(am[2], am[3]));
            const float amax = warp_max_f32(fmaxf(__low2float(m2), __high2float(m2)));
            const float sc = __fdiv_rn(amax, 127.0f);
            if (lane == 0) srow[k.q] = sc;
            const float inv = quant_reciprocal(sc);
            uint2* dst = reinterpret_cast<uint2*>(a.codes[k.q] + k.j0);
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const uint4 wv = src[v * 32 + lane];
                const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
                uint32_t packed[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float xs[4] = {Lp<ZERO_BF16>::lo(ws[2 * h]), Lp<ZERO_BF16>::hi(ws[2 * h]),
                                         Lp<ZERO_BF16>::lo(ws[2 * h + 1]), Lp<ZERO_BF16>::hi(ws[2 * h + 1])};
                    float cf[4];
                    packed[h] = quant_code4(xs, sc, inv, cf);
                }
                dst[v * 32 + lane] = make_uint2(packed[0], packed[1]);
            }
            // every lane's reads of the slot are complete (their values were used): refill it
            __syncwarp();
            issue(s);
        } else {
            issue(s);
            const uint16_t* x = a.rank[k.q] + k.j0;
            float amax = 0.0f;
            for (int i = lane; i < k.n; i += 32) amax = fmaxf(amax, fabsf(Lp<ZERO_BF16>::widen(x[i])));
            amax = warp_max_f32(amax);
            const float sc = __fdiv_rn(amax, 127.0f);
            if (lane == 0) srow[k.q] = sc;
            const float inv = quant_reciprocal(sc);
            signed char* c = a.codes[k.q] + k.j0;
            for (int i = lane; i < k.n; i += 32) c[i] = quant_code(Lp<ZERO_BF16>::widen(x[i]), sc, inv);
        }
    }
    if (!ok && lane == 0) {
        // a wait ran out: let the copies in flight land before the CTA's
        // shared memory is released, then report
        for (int s = 0; s < kQsSlots; ++s)
            if (pending & (1u << s)) mbar_wait_bounded(&bar[s], (phase >> s) & 1u, nullptr, a.timeout_ns);
        if (a.sc != nullptr) atomicOr(&a.sc->status, ZERO_DEV_TIMEOUT);
    }
}

cudaError_t launch_quantize_grads(const void* const* ranks, int n_d, long long shard, long long psi, int block,
                                  signed char* const* codes, float* scales, zero_dev_scalars* sc, cudaStream_t st,
                                  bool starve)
{
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    QsArgs a;
    std::memset(&a, 0, sizeof(a));
    bool aligned = true;
    for (int q = 0; q < n_d; ++q) {
        a.rank[q] = static_cast<const uint16_t*>(ranks[q]);
        a.codes[q] = codes[q];
        aligned = aligned && (reinterpret_cast<uintptr_t>(ranks[q]) & 15) == 0 &&
                  (reinterpret_cast<uintptr_t>(codes[q]) & 15) == 0;
    }
    a.scales = scales;
    a.sc = sc;
    a.shard = shard;
    a.psi = psi;
    a.block = block;
    a.n_d = n_d;
    a.nbs = (shard + block - 1) / block;
    a.n_dp = (n_d + 3) / 4 * 4;
    a.total = static_cast<long long>(n_d) * n_d * a.nbs;
    if (a.nbs > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    a.ring_ok = (block == kQuantBlock && shard % 8 == 0 && aligned) ? 1 : 0;
    a.timeout_ns = starve ? 2000000ull : kDefaultTimeoutNs;
    a.starve = starve ? 1 : 0;
    if (a.total <= 0) return cudaSuccess;
    const size_t smem = 1024 + static_cast<size_t>(kQsWarps) * kQsSlots * kQsSlotBytes;
    static int attr_done[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !__atomic_load_n(&attr_done[dev], __ATOMIC_ACQUIRE)) {
        const cudaError_t e =
            cudaFuncSetAttribute(k_quantize_ranks, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        __atomic_store_n(&attr_done[dev], 1, __ATOMIC_RELEASE);
    }
    long long grid = (a.total + kQsWarps - 1) / kQsWarps;
    if (grid > sms) grid = sms;
    count_launch();
    k_quantize_ranks<<<static_cast<unsigned>(grid), kQsWarps * 32, smem, st>>>(a);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- diagnostics
// Waits on a barrier that nothing completes until the limit runs out, then
// reports ZERO_DEV_TIMEOUT and returns.
__global__ void k_debug_wait(zero_dev_scalars* sc, unsigned long long timeout_ns)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
        if (!mbar_wait_bounded(&bar, 0u, nullptr, timeout_ns)) atomicOr(&sc->status, ZERO_DEV_TIMEOUT);
    }
}

cudaError_t launch_debug_wait(zero_dev_scalars* sc, unsigned long long timeout_ns, cudaStream_t st)
{
    count_launch();
    k_debug_wait<<<1, 32, 0, st>>>(sc, timeout_ns);
    return cudaGetLastError();
}

}  // namespace zk
