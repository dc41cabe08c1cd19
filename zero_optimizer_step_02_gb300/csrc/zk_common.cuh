// zk_common.cuh -- device helpers shared by the libzero kernels (sm_103a).
//
// PTX wrappers for mbarriers and 1-D bulk (TMA) copies, bounded waits,
// 16-bit float conversions and the per-step Adam constants.  All floating
// point that decides a result is written with explicit round-to-nearest
// intrinsics so that no multiply-add is contracted and every operation is one
// IEEE rounding, in the order the update rule states.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "zero.h"

namespace zk {

// ------------------------------------------------------------------ geometry
constexpr int kTile = 4096;                 // elements per tile of the streaming engine
constexpr int kConsumerWarps = 16;         // one 4-element chunk per consumer thread per tile
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;   // + one producer warp
constexpr int kChunk = 4;                   // consecutive elements per consumer chunk
constexpr int kChunksPerThread = kTile / (kChunk * kConsumers);
static_assert(kChunksPerThread * kChunk * kConsumers == kTile, "tile / consumer mismatch");
constexpr int kQuantBlock = kChunk * kConsumers;  // fused int8 gather: one block per chunk row (2048)
constexpr int kGroupRanks = 8;              // rank slices per pipeline stage
constexpr int kMaxSide = 4;                 // fp32 side streams (g, master, m, v)
constexpr int kMaxStages = 8;
// Ring depth the engine uses with its state in HBM: two stages measured
// faster than three for every op (the clipped GPT-2-small step 0.980 ->
// 0.940 ms); 152 SMs x 2 stages of up to 112 KB already keep ~20-34 MB in
// flight, and more only adds L2 and DRAM contention.  With the state in host
// memory the ring stages only the small reduced-gradient tiles and keeps the
// deeper ring (up to kMaxStages), which that path measured faster with; so
// does the fused step over several groups of int8 ranks, whose state is read
// directly (the stages then hold codes only: three of 64 KB fit).
constexpr int kRingStages = 2;
constexpr int kStageOffset = 1024;          // dynamic smem bytes before the stage ring
constexpr int kMaxPartials = 4096;          // per-CTA partial sums kept in the workspace
constexpr unsigned long long kDefaultTimeoutNs = 4000000000ull;  // 4 s per wait

// flags of a streaming launch
enum : int {
    F_GUARD = 1 << 0,   // skip the whole kernel if scalars->nonfinite is set
    F_DETECT = 1 << 1,  // OR "non-finite reduced gradient" into scalars->nonfinite
    F_SQNORM = 1 << 2,  // per-CTA partial sums of the squared reduced gradient
    F_CLIP = 1 << 3,    // multiply the gradient by scalars->clip_coef
    F_QUANT = 1 << 4,   // fused block-int8 quantized gather epilogue
    F_LSCALE = 1 << 5,  // divisor includes scalars->loss_scale
    F_FINALIZE = 1 << 6,  // every CTA sums the reduce pass's partials itself (clip coefficient)
    F_EPILOGUE = 1 << 7,  // the last CTA to finish commits the step scalars
    F_REVERSE = 1 << 8,   // flat launches: walk the tiles from the end (reads what the
                          // previous pass wrote last first, while it is still in L2)
    F_CARRY = 1 << 9,     // gradient accumulation: the rank sum is added to an fp32 carry
                          // stream (side 0 of OP_REDUCE, side 3 of OP_FUSED) before the mean
    F_RAW = 1 << 10,      // OP_REDUCE: store the sum itself, no division
    F_DEBUG_STARVE = 1 << 11,   // the producer issues no copy, so every consumer wait
                                // runs out (tests the timeout path; nothing is read)
    F_HOST_STATE = 1 << 12,     // master/m/v in page-locked host memory (launch shape only)
};

// ------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// make barrier initialisation visible to the async (bulk copy) proxy
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// order this thread's earlier shared-memory accesses before later bulk copies
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One test of the phase; while it is incomplete the thread is suspended in
// hardware until it completes or kWaitHintNs pass, so a waiting warp does not
// spin on issue slots the working warps need.
constexpr uint32_t kWaitHintNs = 10000000u;

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kWaitHintNs)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of `bar` with the given parity.  Bounded twice: by a
// wall-clock limit and by an iteration count.  Returns false when the limit
// ran out or another thread of the CTA raised *abort.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  const volatile int* abort,
                                                  unsigned long long timeout_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1; it < (1u << 28); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        // each test may have slept up to kWaitHintNs: check every time
        if (abort != nullptr && *abort) return false;
        if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
    return false;
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.  (An L2
// evict-first hint on these streamed loads measured no better, or worse.)
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                          uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1], %2, [%3];" ::"r"(smem_u32(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 1-D bulk copy shared -> global, tracked by bulk async-groups.
__device__ __forceinline__ void bulk_store(void* gmem_dst, const void* smem_src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
                 "r"(smem_u32(smem_src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// wait until at most N bulk groups still read shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_all()
{
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// -------------------------------------------------------- 16-bit encodings
template <int DT>
struct Lp;

// ------------------------------------------- packed and mixed fp32 arithmetic
// sm_100-family instructions that do what several scalar ones do, with the
// same IEEE round-to-nearest results (subnormals kept): an fp32 add of a
// 16-bit operand (the widening is exact, so this is fadd(widen(h), acc)),
// and fp32 operations on register pairs.  Caution: ptxas fuses a packed
// multiply that feeds a packed add or subtract into one rounding, whatever
// the rounding modifier or -fmad setting; packed multiplies are used only
// where that cannot change a result (the quantizer's fast path).
__device__ __forceinline__ void halves(uint32_t w, unsigned short& lo, unsigned short& hi)
{
    asm("mov.b32 {%0, %1}, %2;" : "=h"(lo), "=h"(hi) : "r"(w));
}
__device__ __forceinline__ float add_bf16_f32(unsigned short h, float acc)
{
    float d;
    asm("add.rn.f32.bf16 %0, %1, %2;" : "=f"(d) : "h"(h), "f"(acc));
    return d;
}
__device__ __forceinline__ float add_f16_f32(unsigned short h, float acc)
{
    float d;
    asm("add.rn.f32.f16 %0, %1, %2;" : "=f"(d) : "h"(h), "f"(acc));
    return d;
}
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pack2(float a, float b)
{
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void unpack2(f32x2 v, float& a, float& b)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b)
{
    f32x2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b)
{
    f32x2 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b)
{
    f32x2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

template <>
struct Lp<ZERO_BF16> {
    // acc + the 16-bit value h, one rounding
    __device__ static __forceinline__ float add(float acc, unsigned short h) { return add_bf16_f32(h, acc); }
    // a 32-bit word holds two consecutive elements, the first in the low half
    __device__ static __forceinline__ float lo(uint32_t w) { return __uint_as_float(w << 16); }
    __device__ static __forceinline__ float hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
    __device__ static __forceinline__ float widen(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }
    __device__ static __forceinline__ uint16_t narrow(float x)
    {
        return __bfloat16_as_ushort(__float2bfloat16_rn(x));
    }
    // two values in one conversion, a in the low half (each rounded as narrow)
    __device__ static __forceinline__ uint32_t narrow2(float a, float b)
    {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
};

template <>
struct Lp<ZERO_FP16> {
    __device__ static __forceinline__ float add(float acc, unsigned short h) { return add_f16_f32(h, acc); }
    __device__ static __forceinline__ float lo(uint32_t w)
    {
        return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
    }
    __device__ static __forceinline__ float hi(uint32_t w)
    {
        return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
    }
    __device__ static __forceinline__ float widen(uint16_t h) { return __half2float(__ushort_as_half(h)); }
    __device__ static __forceinline__ uint16_t narrow(float x) { return __half_as_ushort(__float2half_rn(x)); }
    __device__ static __forceinline__ uint32_t narrow2(float a, float b)
    {
        const __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
};

__device__ __forceinline__ bool is_finite_f32(float x)
{
    return (__float_as_uint(x) & 0x7F800000u) != 0x7F800000u;
}

// ------------------------------------------------------------ step constants
// Everything a kernel needs from the hyper-parameters and the step scalars,
// computed once per CTA by one thread.
struct StepConsts {
    float b1, b2, omb1, omb2, step, eps, decay, coef;   // step, eps: bias-corrected (see set_adam)
    float divisor, inv_divisor;
    int wd, clip, div_pow2;
};

// The divisor of the mean: n_d times the loss scale (when loss scaling).
// When it is a power of two, x * (1/D) is the same correctly rounded value as
// x / D (both round the same real number), so the multiply is used.
__device__ __forceinline__ void set_divisor(StepConsts& c, int n_d, float loss_scale)
{
    c.divisor = __fmul_rn(static_cast<float>(n_d), loss_scale);
    const uint32_t b = __float_as_uint(c.divisor);
    const uint32_t e = (b >> 23) & 0xFFu;
    c.div_pow2 = (b & 0x007FFFFFu) == 0 && e != 0 && e != 0xFFu && (b >> 31) == 0;
    c.inv_divisor = c.div_pow2 ? __frcp_rn(c.divisor) : 0.0f;
}

// Bias-corrected Adam constants for the step about to be committed: the fp64
// running products beta^t are extended by one multiplication (never pow).
// Adam in the order Kingma & Ba give as the efficient form of their
// Algorithm 1: step = lr * sqrt(1 - beta2^t) / (1 - beta1^t) and
// eps_hat = eps * sqrt(1 - beta2^t), equal to Algorithm 1 in exact
// arithmetic, with one division per element instead of two.
__device__ __forceinline__ void set_adam(StepConsts& c, const zero_hparams& hp, double b1pow,
                                         double b2pow)
{
    const double b1t = __dmul_rn(b1pow, static_cast<double>(hp.beta1));
    const double b2t = __dmul_rn(b2pow, static_cast<double>(hp.beta2));
    const float bc1 = __double2float_rn(__dsub_rn(1.0, b1t));
    const float bc2 = __double2float_rn(__dsub_rn(1.0, b2t));
    const float sbc2 = __fsqrt_rn(bc2);
    c.b1 = hp.beta1;
    c.b2 = hp.beta2;
    c.omb1 = __fsub_rn(1.0f, hp.beta1);
    c.omb2 = __fsub_rn(1.0f, hp.beta2);
    c.step = __fdiv_rn(__fmul_rn(hp.lr, sbc2), bc1);
    c.eps = __fmul_rn(hp.eps, sbc2);
    c.decay = __fsub_rn(1.0f, __fmul_rn(hp.lr, hp.weight_decay));
    c.wd = hp.weight_decay != 0.0f;
}

__device__ __forceinline__ float mean_of(const StepConsts& c, float sum)
{
    return c.div_pow2 ? __fmul_rn(sum, c.inv_divisor) : __fdiv_rn(sum, c.divisor);
}

// The mean of four sums: the divisor's form is tested once for the four.
// With a power-of-two divisor the mean is an exact multiplication, done on
// register pairs (the products feed only multiplications and stores, so
// nothing can be contracted into them).
__device__ __forceinline__ void mean_of4(const StepConsts& c, const float (&sum)[4], float (&g)[4])
{
    if (c.div_pow2) {
        const f32x2 inv = pack2(c.inv_divisor, c.inv_divisor);
        unpack2(mul2(pack2(sum[0], sum[1]), inv), g[0], g[1]);
        unpack2(mul2(pack2(sum[2], sum[3]), inv), g[2], g[3]);
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) g[e] = __fdiv_rn(sum[e], c.divisor);
    }
}

// Four Adam/AdamW element updates, each in adam_elem's operation order; the
// weight-decay test is made once for the four.
__device__ __forceinline__ void adam_elem4(const StepConsts& c, const float (&g)[4], float (&p)[4], float (&m)[4],
                                           float (&v)[4])
{
    if (c.wd) {
#pragma unroll
        for (int e = 0; e < 4; ++e) p[e] = __fmul_rn(p[e], c.decay);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        m[e] = __fadd_rn(__fmul_rn(c.b1, m[e]), __fmul_rn(c.omb1, g[e]));
        v[e] = __fadd_rn(__fmul_rn(c.b2, v[e]), __fmul_rn(c.omb2, __fmul_rn(g[e], g[e])));
        const float denom = __fadd_rn(__fsqrt_rn(v[e]), c.eps);
        p[e] = __fsub_rn(p[e], __fmul_rn(c.step, __fdiv_rn(m[e], denom)));
    }
}

// One Adam/AdamW element update in the fixed operation order.
__device__ __forceinline__ void adam_elem(const StepConsts& c, float g, float& p, float& m, float& v)
{
    if (c.wd) p = __fmul_rn(p, c.decay);
    m = __fadd_rn(__fmul_rn(c.b1, m), __fmul_rn(c.omb1, g));
    v = __fadd_rn(__fmul_rn(c.b2, v), __fmul_rn(c.omb2, __fmul_rn(g, g)));
    const float denom = __fadd_rn(__fsqrt_rn(v), c.eps);
    p = __fsub_rn(p, __fmul_rn(c.step, __fdiv_rn(m, denom)));
}

// Squared-norm accumulation with an error-free product and a compensated sum
// in fp32 (the per-thread partial is then carried in fp64): the result agrees
// with an fp64 sum of the exact squares to ~1e-14 relative, so the clipping
// coefficient comes out the same as a sequential fp64 sum's.  Every term and
// the running sum are non-negative, so ordering the pair by max / min makes
// Dekker's Fast2Sum (s = a + b, e = b - (s - a), exact for a >= b >= 0) do
// what Knuth's TwoSum does, with one floating-point operation fewer and the
// ordering on the integer-side pipe.  Adding g = 0 changes nothing (hi stays,
// e = 0), so padding past a tile's valid length needs no test.
__device__ __forceinline__ void sq_accumulate(float g, float& hi, float& lo)
{
    const float p = __fmul_rn(g, g);
    const float pe = __fmaf_rn(g, g, -p);
    const float a = fmaxf(hi, p);
    const float b = fminf(hi, p);
    const float s = __fadd_rn(a, b);
    const float e = __fsub_rn(b, __fsub_rn(s, a));
    hi = s;
    lo = __fadd_rn(lo, __fadd_rn(e, pe));
}

__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c)
{
    f32x2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// sq_accumulate on two elements at once, into two compensated sums (the even
// and the odd elements of a chunk) on register pairs: the same per-sum
// arithmetic with one instruction for two of each add, subtract, multiply and
// FMA (the clipped GPT-2-small step with int8 gradients 0.4% faster)
__device__ __forceinline__ void sq_accumulate2(float g0, float g1, f32x2& hi, f32x2& lo)
{
    const f32x2 g = pack2(g0, g1);
    const f32x2 p = mul2(g, g);
    float p0, p1, h0, h1;
    unpack2(p, p0, p1);
    unpack2(hi, h0, h1);
    const f32x2 pe = fma2(g, g, pack2(-p0, -p1));
    const f32x2 a = pack2(fmaxf(h0, p0), fmaxf(h1, p1));
    const f32x2 b = pack2(fminf(h0, p0), fminf(h1, p1));
    const f32x2 s = add2(a, b);
    const f32x2 e = sub2(b, sub2(s, a));
    hi = s;
    lo = add2(lo, add2(e, pe));
}

// Clip coefficient of the clipping reading: max_norm / (norm + 1e-6) when
// that is below one, else 1 (and 1 when clipping is off).
__device__ __forceinline__ float clip_coefficient(float max_norm, double sqnorm)
{
    if (!(max_norm > 0.0f)) return 1.0f;
    const double norm = __dsqrt_rn(sqnorm);
    const float c = __double2float_rn(__ddiv_rn(static_cast<double>(max_norm), __dadd_rn(norm, 1e-6)));
    return c < 1.0f ? c : 1.0f;
}

// Commit (or skip) the step, per the loss-scaling reading: a step whose
// reduced gradient held a non-finite value leaves the state alone, halves
// the scale (floor min_scale) and resets the good-step count; otherwise t
// advances, the beta powers take one more factor, and after scale_window
// good steps the scale doubles.  Clears the step's non-finite flag.
__device__ __forceinline__ void commit_scalars(const zero_hparams& hp, zero_dev_scalars* sc)
{
    const bool skip = hp.loss_scaling && *reinterpret_cast<volatile int*>(&sc->nonfinite) != 0;
    if (skip) {
        const float half = __fmul_rn(sc->loss_scale, 0.5f);
        sc->loss_scale = half > hp.min_scale ? half : hp.min_scale;
        sc->good_steps = 0;
        sc->overflow = 1;
        sc->clip_coef = 1.0f;
    } else {
        sc->t += 1;
        sc->beta1_pow = __dmul_rn(sc->beta1_pow, static_cast<double>(hp.beta1));
        sc->beta2_pow = __dmul_rn(sc->beta2_pow, static_cast<double>(hp.beta2));
        sc->overflow = 0;
        if (hp.loss_scaling) {
            sc->good_steps += 1;
            if (sc->good_steps >= hp.scale_window) {
                sc->loss_scale = __fmul_rn(sc->loss_scale, 2.0f);
                sc->good_steps = 0;
            }
        }
    }
    if (!(hp.max_norm > 0.0f)) {
        sc->sqnorm = 0.0;
        sc->clip_coef = 1.0f;
    }
    sc->nonfinite = 0;
}

// ------------------------------------------------------------- quantizer
// Block-int8 code of x with scale s: clamp(round-half-even(x / s), -127, 127),
// 0 when s == 0, where x / s is the IEEE-rounded quotient.  The quotient only
// feeds a rounding to an integer, so x * (1/s) is used instead, and the exact
// quotient only when that product lies within 2^-14 of a half-integer: the
// product and the quotient differ by a few ulp of a value below 128 (an ulp
// there is at most 2^-17), so away from a tie both round to the same integer.
// inv = quant_reciprocal(s); 0 unless s is a positive normal float below
// 3e38 (then every code takes the exact quotient).  With a normal s,
// |x * inv| <= 127 (1 + 2^-22) for every |x| <= amax, so the fast codes
// never need the clamp.
__device__ __forceinline__ float quant_reciprocal(float s)
{
    if (!(s >= 1.17549435e-38f) || !(s < 3.0e38f)) return 0.0f;
    return __frcp_rn(s);
}

// Round to nearest, ties to even, with one addition: for |y| < 2^22,
// y + 1.5 * 2^23 keeps no fraction bits, so the sum is rint(y) + 1.5 * 2^23
// exactly and subtracting the constant gives rint(y); the sum's low byte is
// the two's-complement low byte of rint(y) (the constant's low 22 bits are
// zero).  Larger |y| are not rounded exactly but stay beyond +-127.5, which
// the clamp below maps to +-127 as it would rint(y); NaN clamps to -127 as
// fmaxf(rintf(NaN), -127) does.  Full-rate FP adds instead of the conversion
// unit's rint / floor / float-to-int.
constexpr float kRintShift = 12582912.0f;
// |y - rint(y)| at or above this: y lies within 2^-14 of a half-integer
constexpr float kTieBand = 0.49993896484375f;   // 0.5 - 2^-14

__device__ __forceinline__ float rint_shift(float y) { return __fsub_rn(__fadd_rn(y, kRintShift), kRintShift); }

__device__ __forceinline__ float clamp127(float r) { return fminf(fmaxf(r, -127.0f), 127.0f); }

// the int8 bits of an integer-valued float in [-127, 127], in the low byte
__device__ __forceinline__ uint32_t code_bits(float cf) { return __float_as_uint(__fadd_rn(cf, kRintShift)); }

// Codes of four values at once: the fast products for all four, and one
// (rarely taken) branch to the exact quotients if any of them is near a tie.
// cf receives the codes as floats (for dequantization); the return value
// packs the four int8 codes, code e in byte e.
__device__ __forceinline__ uint32_t quant_code4(const float (&x)[4], float s, float inv, float (&cf)[4])
{
    if (s == 0.0f) {
#pragma unroll
        for (int e = 0; e < 4; ++e) cf[e] = 0.0f;
        return 0u;
    }
    // fast: t = rint(x * inv) + 1.5 * 2^23 (its low byte is the code), no
    // clamp needed (see quant_reciprocal); a NaN product fails the test below.
    // The packed multiply may be fused into the adds (one rounding of the
    // exact product P): away from the tie band rint(P) is still the integer
    // the exact quotient rounds to (|P - x/s| < 2^-17, band 2^-14), and in
    // it the exact quotient decides.
    float t[4], d[4];
    {
        const f32x2 inv2 = pack2(inv, inv), m2 = pack2(kRintShift, kRintShift);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const f32x2 y = mul2(pack2(x[2 * h], x[2 * h + 1]), inv2);
            const f32x2 tt = add2(y, m2);
            const f32x2 c = sub2(tt, m2);
            unpack2(tt, t[2 * h], t[2 * h + 1]);
            unpack2(c, cf[2 * h], cf[2 * h + 1]);
            unpack2(sub2(y, c), d[2 * h], d[2 * h + 1]);
        }
    }
    bool near = inv == 0.0f;
#pragma unroll
    for (int e = 0; e < 4; ++e) near |= !(fabsf(d[e]) < kTieBand);
    if (near) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            cf[e] = clamp127(rint_shift(__fdiv_rn(x[e], s)));
            t[e] = __fadd_rn(cf[e], kRintShift);
        }
    }
    const uint32_t u[4] = {__float_as_uint(t[0]), __float_as_uint(t[1]), __float_as_uint(t[2]), __float_as_uint(t[3])};
    return __byte_perm(__byte_perm(u[0], u[1], 0x0040u), __byte_perm(u[2], u[3], 0x0040u), 0x5410u);
}

// One code, as a float (see quant_code4).
__device__ __forceinline__ float quant_code_f(float x, float s, float inv)
{
    if (s == 0.0f) return 0.0f;
    if (inv != 0.0f) {
        const float y = __fmul_rn(x, inv);
        const float r = rint_shift(y);
        if (fabsf(__fsub_rn(y, r)) < kTieBand) return r;   // else near a tie (or NaN): decide exactly
    }
    return clamp127(rint_shift(__fdiv_rn(x, s)));
}

__device__ __forceinline__ int8_t quant_code(float x, float s, float inv)
{
    return static_cast<int8_t>(static_cast<uint8_t>(code_bits(quant_code_f(x, s, inv))));
}

__device__ __forceinline__ double warp_sum_f64(double x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = __dadd_rn(x, __shfl_xor_sync(0xFFFFFFFFu, x, o));
    return x;
}

__device__ __forceinline__ float warp_max_f32(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xFFFFFFFFu, x, o));
    return x;
}

}  // namespace zk
