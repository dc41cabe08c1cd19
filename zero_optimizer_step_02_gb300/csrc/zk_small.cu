// zk_small.cu -- the fused step for problems too small to fill the streaming
// engine's pipeline.
//
// One thread per 4 consecutive elements: the ranks' 16-bit gradients, the
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

template <int GT, int PT>
__global__ void __launch_bounds__(kSmallThreads) k_small_step(const __grid_constant__ SmallArgs a)
{
    __shared__ StepConsts shc;
    zero_dev_scalars* sc = a.sc;
    if (threadIdx.x == 0) {
        StepConsts c = {};
        set_divisor(c, a.n_ranks, 1.0f);
        set_adam(c, a.hp, sc->beta1_pow, sc->beta2_pow);
        c.clip = 0;
        c.coef = 1.0f;
        shc = c;
    }
    __syncthreads();
    const StepConsts c = shc;
    const long long j = a.lo + 4LL * (static_cast<long long>(blockIdx.x) * kSmallThreads + threadIdx.x);
    if (j < a.hi) {
        const int cnt = a.hi - j >= 4 ? 4 : static_cast<int>(a.hi - j);
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f}, p[4], m[4], v[4];
        if (cnt == 4) {
            // j is a multiple of 4 from a 16-byte aligned start: 8-byte
            // rank words, 16-byte state vectors
            for (int r = 0; r < a.n_ranks; ++r)
                add4<GT>(acc, *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a.rank[r]) + j));
            const float4 fp = *reinterpret_cast<const float4*>(a.master_in + j);
            const float4 fm = *reinterpret_cast<const float4*>(a.m_in + j);
            const float4 fv = *reinterpret_cast<const float4*>(a.v_in + j);
            p[0] = fp.x; p[1] = fp.y; p[2] = fp.z; p[3] = fp.w;
            m[0] = fm.x; m[1] = fm.y; m[2] = fm.z; m[3] = fm.w;
            v[0] = fv.x; v[1] = fv.y; v[2] = fv.z; v[3] = fv.w;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                p[e] = m[e] = v[e] = 0.0f;
                if (e < cnt) {
                    for (int r = 0; r < a.n_ranks; ++r)
                        acc[e] = Lp<GT>::add(acc[e], static_cast<const uint16_t*>(a.rank[r])[j + e]);
                    p[e] = a.master_in[j + e];
                    m[e] = a.m_in[j + e];
                    v[e] = a.v_in[j + e];
                }
            }
        }
        float g[4];
        mean_of4(c, acc, g);
        adam_elem4(c, g, p, m, v);
        uint16_t lp[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) lp[e] = Lp<PT>::narrow(p[e]);
        if (cnt == 4) {
            *reinterpret_cast<float4*>(a.master_out + j) = make_float4(p[0], p[1], p[2], p[3]);
            *reinterpret_cast<float4*>(a.m_out + j) = make_float4(m[0], m[1], m[2], m[3]);
            *reinterpret_cast<float4*>(a.v_out + j) = make_float4(v[0], v[1], v[2], v[3]);
            if (a.lp_out != nullptr) {
                uint2 w;
                w.x = static_cast<uint32_t>(lp[0]) | (static_cast<uint32_t>(lp[1]) << 16);
                w.y = static_cast<uint32_t>(lp[2]) | (static_cast<uint32_t>(lp[3]) << 16);
                *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.lp_out) + j) = w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (e < cnt) {
                    a.master_out[j + e] = p[e];
                    a.m_out[j + e] = m[e];
                    a.v_out[j + e] = v[e];
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

cudaError_t launch_small_step(int grad_dtype, int param_dtype, const SmallArgs& a, cudaStream_t st)
{
    const long long n = a.hi - a.lo;
    if (n <= 0) return cudaSuccess;
    const long long threads = (n + 3) / 4;
    const unsigned grid = static_cast<unsigned>((threads + kSmallThreads - 1) / kSmallThreads);
    count_launch();
    const bool gb = grad_dtype == ZERO_BF16, pb = param_dtype == ZERO_BF16;
    if (gb && pb) k_small_step<ZERO_BF16, ZERO_BF16><<<grid, kSmallThreads, 0, st>>>(a);
    else if (gb) k_small_step<ZERO_BF16, ZERO_FP16><<<grid, kSmallThreads, 0, st>>>(a);
    else if (pb) k_small_step<ZERO_FP16, ZERO_BF16><<<grid, kSmallThreads, 0, st>>>(a);
    else k_small_step<ZERO_FP16, ZERO_FP16><<<grid, kSmallThreads, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace zk
