// zk_small.cu -- the fused step for problems too small to fill the streaming
// engine's pipeline.
//
// One thread per 4 consecutive elements (two such chunks when the step's
// threads would not all fit on the GPU at once): the ranks' 16-bit gradients, the
// fp32 master/m/v and the 16-bit results move with plain 8- and 16-byte loads
// and stores, straight between HBM (or L2) and registers, with many CTAs per
// SM and no staging, so every load of the step is in flight at once and
// nothing waits for a pipeline to fill.  The arithmetic is the engine's fused
// step, operation for operation (the rank-ordered fp32 sum from +0, the mean,
// Adam in the order of the update rule, the round-to-nearest-even cast), so
// the results are the same bits.
//
// Used for the plain fused step (no clipping, no loss scaling, no
// accumulation carry, state in device memory) when the engine would have
// fewer than two 4096-element tiles per SM.  Sources: DP-notes "ZeRO-2:
// Gradient Partitioning" (reduce-scatter, then each rank updates its own
// partition); itwiki "FSDP와의 관계" (fp32 reduce).
#include "zk_common.cuh"
#include "zk_launch.h"

namespace zk {

namespace {

constexpr int kSmallThreads = 256;
// gradient words of this many ranks are loaded before the first is added, so
// their DRAM latencies overlap instead of following one another
constexpr int kRankGroup = 4;

// the four 16-bit values of an 8-byte word added to acc, one rounding each
template <int GT>
__device__ __forceinline__ void add4(float (&acc)[4], uint2 w)
{
    unsigned short h[4];
    halves(w.x, h[0], h[1]);
    halves(w.y, h[2], h[3]);
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[e] = Lp<GT>::add(acc[e], h[e]);
}

// one rank's 16-bit gradients of elements [j, j + cnt) as an 8-byte word
// (zeros past cnt; those lanes are never stored)
__device__ __forceinline__ uint2 load_grads(const void* rank, long long j, int cnt)
{
    const uint16_t* g = static_cast<const uint16_t*>(rank) + j;
    if (cnt == 4) return *reinterpret_cast<const uint2*>(g);
    uint32_t h[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int e = 0; e < 4; ++e)
        if (e < cnt) h[e] = g[e];
    return make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
}

// at most 48 registers with one chunk (5 CTAs per SM), 64 with two (4 CTAs:
// the largest problem given to this kernel, 2 x 152 x 4096 elements, then
// fits on the GPU at once)
template <int GT, int PT, int kChunks>
__global__ void __launch_bounds__(kSmallThreads, kChunks == 1 ? 5 : 4) k_small_step(const __grid_constant__ SmallArgs a)
{
    __shared__ StepConsts shc;
    zero_dev_scalars* sc = a.sc;
    // Thread 0's read of the step scalars goes out first, ahead of the data
    // (behind 20 MB of requests it would come back last); then chunk k of
    // this thread, elements [4 (t0 + k * nth), + 4): every chunk's master/m/v
    // and its first kRankGroup ranks' gradients are loaded before anything
    // waits on them, and thread 0 forms the constants while they are in flight
    double b1pow = 0.0, b2pow = 0.0;
    if (threadIdx.x == 0) {
        b1pow = sc->beta1_pow;
        b2pow = sc->beta2_pow;
    }
    const long long nth = static_cast<long long>(gridDim.x) * kSmallThreads;
    const long long t0 = static_cast<long long>(blockIdx.x) * kSmallThreads + threadIdx.x;
    const int g0 = a.n_ranks < kRankGroup ? a.n_ranks : kRankGroup;
    float acc[kChunks][4], p[kChunks][4], m[kChunks][4], v[kChunks][4];
    uint2 w[kChunks][kRankGroup];
    int cnt[kChunks];
    long long jj[kChunks];
#pragma unroll
    for (int k = 0; k < kChunks; ++k) {
        const long long j = a.lo + 4LL * (t0 + k * nth);
        jj[k] = j;
        cnt[k] = j >= a.hi ? 0 : (a.hi - j >= 4 ? 4 : static_cast<int>(a.hi - j));
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[k][e] = p[k][e] = m[k][e] = v[k][e] = 0.0f;
#pragma unroll
        for (int r = 0; r < kRankGroup; ++r) {
            w[k][r] = make_uint2(0u, 0u);
            if (r < g0 && cnt[k] > 0) w[k][r] = load_grads(a.rank[r], j, cnt[k]);
        }
        if (cnt[k] == 4) {
            const float4 fp = *reinterpret_cast<const float4*>(a.master_in + j);
            const float4 fm = *reinterpret_cast<const float4*>(a.m_in + j);
            const float4 fv = *reinterpret_cast<const float4*>(a.v_in + j);
            p[k][0] = fp.x; p[k][1] = fp.y; p[k][2] = fp.z; p[k][3] = fp.w;
            m[k][0] = fm.x; m[k][1] = fm.y; m[k][2] = fm.z; m[k][3] = fm.w;
            v[k][0] = fv.x; v[k][1] = fv.y; v[k][2] = fv.z; v[k][3] = fv.w;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (e < cnt[k]) {
                    p[k][e] = a.master_in[j + e];
                    m[k][e] = a.m_in[j + e];
                    v[k][e] = a.v_in[j + e];
                }
            }
        }
    }
    if (threadIdx.x == 0) {
        StepConsts c = {};
        set_divisor(c, a.n_ranks, 1.0f);
        set_adam(c, a.hp, b1pow, b2pow);
        c.clip = 0;
        c.coef = 1.0f;
        shc = c;
    }
    __syncthreads();
    const StepConsts c = shc;
    // the rank-ordered sums from +0: the loaded group, then any further
    // groups, each loaded whole before it is added
#pragma unroll
    for (int k = 0; k < kChunks; ++k)
#pragma unroll
        for (int r = 0; r < kRankGroup; ++r)
            if (r < g0) add4<GT>(acc[k], w[k][r]);
    for (int r0 = kRankGroup; r0 < a.n_ranks; r0 += kRankGroup) {
        const int gn = a.n_ranks - r0 < kRankGroup ? a.n_ranks - r0 : kRankGroup;
#pragma unroll
        for (int k = 0; k < kChunks; ++k)
#pragma unroll
            for (int r = 0; r < kRankGroup; ++r)
                if (r < gn && cnt[k] > 0) w[k][r] = load_grads(a.rank[r0 + r], jj[k], cnt[k]);
#pragma unroll
        for (int k = 0; k < kChunks; ++k)
#pragma unroll
            for (int r = 0; r < kRankGroup; ++r)
                if (r < gn) add4<GT>(acc[k], w[k][r]);
    }
#pragma unroll
    for (int k = 0; k < kChunks; ++k) {
        if (cnt[k] == 0) continue;
        const long long j = jj[k];
        float g[4];
        mean_of4(c, acc[k], g);
        adam_elem4(c, g, p[k], m[k], v[k]);
        uint16_t lp[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) lp[e] = Lp<PT>::narrow(p[k][e]);
        if (cnt[k] == 4) {
            *reinterpret_cast<float4*>(a.master_out + j) = make_float4(p[k][0], p[k][1], p[k][2], p[k][3]);
            *reinterpret_cast<float4*>(a.m_out + j) = make_float4(m[k][0], m[k][1], m[k][2], m[k][3]);
            *reinterpret_cast<float4*>(a.v_out + j) = make_float4(v[k][0], v[k][1], v[k][2], v[k][3]);
            if (a.lp_out != nullptr) {
                uint2 o;
                o.x = static_cast<uint32_t>(lp[0]) | (static_cast<uint32_t>(lp[1]) << 16);
                o.y = static_cast<uint32_t>(lp[2]) | (static_cast<uint32_t>(lp[3]) << 16);
                *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.lp_out) + j) = o;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (e < cnt[k]) {
                    a.master_out[j + e] = p[k][e];
                    a.m_out[j + e] = m[k][e];
                    a.v_out[j + e] = v[k][e];
                    if (a.lp_out != nullptr) static_cast<uint16_t*>(a.lp_out)[j + e] = lp[e];
                }
            }
        }
    }
    if (a.epilogue && threadIdx.x == 0) {
        // the last CTA to take a ticket commits the step scalars: every CTA
        // read them before taking its own (no CTA waits for another)
        __threadfence();
        const unsigned done = atomicAdd(&sc->ctas_done, 1u);
        if (done == gridDim.x - 1) {
            __threadfence();
            commit_scalars(a.hp, sc);
            sc->ctas_done = 0u;
        }
    }
}

}  // namespace

bool small_step_fits(long long n)
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    return n < 2LL * sms * kTile;
}

// One 4-element chunk per thread when the step's threads fit on the GPU at
// once; else two per thread, so that they do again (the 1M-parameter step:
// 13.6 instead of 15.3 us with L2 flushed; 600k parameters keep one chunk,
// 11.4 against 13.1 us with two).
template <int GT, int PT>
cudaError_t launch_small_typed(const SmallArgs& a, long long chunks, cudaStream_t st)
{
    // threads of the one-chunk kernel resident at once, per device (looked up once)
    static long long resident_of[64];
    static int ready[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!__atomic_load_n(&ready[dev], __ATOMIC_ACQUIRE)) {
        int sms = 0, per_sm = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return cudaErrorInvalidDevice;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_small_step<GT, PT, 1>, kSmallThreads, 0) !=
            cudaSuccess)
            return cudaErrorInvalidDevice;
        resident_of[dev] = static_cast<long long>(sms) * per_sm * kSmallThreads;
        __atomic_store_n(&ready[dev], 1, __ATOMIC_RELEASE);
    }
    const long long resident = resident_of[dev];
    count_launch();
    if (chunks <= resident) {
        const unsigned grid = static_cast<unsigned>((chunks + kSmallThreads - 1) / kSmallThreads);
        k_small_step<GT, PT, 1><<<grid, kSmallThreads, 0, st>>>(a);
    } else {
        const long long threads = (chunks + 1) / 2;
        const unsigned grid = static_cast<unsigned>((threads + kSmallThreads - 1) / kSmallThreads);
        k_small_step<GT, PT, 2><<<grid, kSmallThreads, 0, st>>>(a);
    }
    return cudaGetLastError();
}

cudaError_t launch_small_step(int grad_dtype, int param_dtype, const SmallArgs& a, cudaStream_t st)
{
    const long long n = a.hi - a.lo;
    if (n <= 0) return cudaSuccess;
    const long long chunks = (n + 3) / 4;
    const bool gb = grad_dtype == ZERO_BF16, pb = param_dtype == ZERO_BF16;
    if (gb && pb) return launch_small_typed<ZERO_BF16, ZERO_BF16>(a, chunks, st);
    if (gb) return launch_small_typed<ZERO_BF16, ZERO_FP16>(a, chunks, st);
    if (pb) return launch_small_typed<ZERO_FP16, ZERO_BF16>(a, chunks, st);
    return launch_small_typed<ZERO_FP16, ZERO_FP16>(a, chunks, st);
}

}  // namespace zk
