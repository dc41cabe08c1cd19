// zk_stream.cu -- the streaming engine of the ZeRO-DP step and its three ops.
//
// One persistent CTA per SM.  Warp 16 is the producer: one thread issues 1-D
// bulk (TMA) copies of 4096-element tiles into a ring of shared-memory stages,
// each stage holding up to 8 ranks' gradient slices (16 for int8 codes) plus,
// with the last rank group of a tile, the staged fp32 side streams (reduced
// gradient / master / m / v).  Warps 0-15 are consumers: they add the rank
// slices in rank order into fp32 registers, release the stage, then apply the
// op and store the results with 16-byte coalesced stores.  Side streams that
// are not staged (state in host memory, an accumulation carry) are read with
// 16-byte loads issued before the stage wait.  Tiles shorter than 4096 (the
// ragged tail, a shard's last tile) or not 16-byte aligned take a plain-load
// path.
//
//   OP_FUSED  : reduce-scatter + Adam + 16-bit cast (or fused int8 gather)
//   OP_REDUCE : reduce-scatter alone (optional fp32 output, squared-norm
//               partials, non-finite detection), or one micro-batch's
//               undivided rank sum added to an fp32 accumulator
//   OP_ADAM   : Adam from an fp32 reduced gradient + 16-bit cast
//   OP_QFUSED / OP_QADAM : OP_FUSED / OP_ADAM with the fused int8 gather as
//               the epilogue (tiles inside shards, one block per 2048)
//
// Sources: DP-notes "ZeRO-2: Gradient Partitioning" (reduce-scatter, then
// each rank updates its own partition), itwiki "FSDP와의 관계" (fp32
// reduce), itwiki "후속 기법" ZeRO++ row (block-quantized weight gather).
#include "zk_common.cuh"
#include "zk_launch.h"

namespace zk {

struct Shared {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    int issued_parity[kMaxStages];
    int abort;
    int skip;   // a guarded pass whose step is flagged: the CTA writes nothing
    StepConsts c;
    alignas(16) float red_f[2][kChunksPerThread][kConsumerWarps];
    double red_d[kConsumerWarps + 1];
};
static_assert(sizeof(Shared) <= kStageOffset, "shared header too large");

// The step constants of a launch, computed by warp 0 of a CTA into sh->c.
// F_FINALIZE: the whole warp sums the reduce pass's per-CTA partials in the
// order k_finalize uses, so every CTA gets the same bits, and CTA 0 records
// the norm and the coefficient in the step scalars.
__device__ __forceinline__ void step_constants(const StreamArgs& a, Shared* sh, int lane)
{
    double sq = 0.0;
    if (a.flags & F_FINALIZE) {
        for (int i = lane; i < a.fin_n; i += 32) sq = __dadd_rn(sq, a.fin_partials[i]);
        sq = warp_sum_f64(sq);
    }
    if (lane != 0) return;
    StepConsts c = {};
    zero_dev_scalars* sc = a.sc;
    set_divisor(c, (a.n_ranks > 0 ? a.n_ranks : 1) * (a.micro > 0 ? a.micro : 1),
                (a.flags & F_LSCALE) ? sc->loss_scale : 1.0f);
    if (sc != nullptr) set_adam(c, a.hp, sc->beta1_pow, sc->beta2_pow);   // null: plain sums only
    c.clip = (a.flags & F_CLIP) != 0;
    if (a.flags & F_FINALIZE) {
        const float coef = clip_coefficient(a.hp.max_norm, sq);
        c.coef = c.clip ? coef : 1.0f;
        if (blockIdx.x == 0) {
            sc->sqnorm = sq;
            sc->clip_coef = coef;
        }
    } else {
        c.coef = c.clip ? sc->clip_coef : 1.0f;
    }
    sh->c = c;
}

// rank-group shapes of a launch (the FULL parameter of k_stream); kFullHalf:
// the int8-rank reduce pass only, one group holding exactly half the slots
// (N_d = 8)
enum { kPartial = 0, kFullOne = 1, kFullMulti = 2, kFullHalf = 3 };

// Walks this CTA's tiles (blockIdx.x, + gridDim.x, ...) as (segment, tile in
// segment) without a 64-bit division per tile: one division at the start,
// then an add-and-carry per step.
struct TileCursor {
    long long seg, t;        // current tile = seg * tiles_per_seg + t
    long long dseg, dt;      // gridDim.x split the same way

    __device__ __forceinline__ void start(const StreamArgs& a)
    {
        const long long first = blockIdx.x, step = gridDim.x;
        seg = first / a.tiles_per_seg;
        t = first - seg * a.tiles_per_seg;
        dseg = step / a.tiles_per_seg;
        dt = step - dseg * a.tiles_per_seg;
    }
    __device__ __forceinline__ bool valid(const StreamArgs& a) const { return seg < a.n_seg; }
    __device__ __forceinline__ void next(const StreamArgs& a)
    {
        seg += dseg;
        t += dt;
        if (t >= a.tiles_per_seg) {
            t -= a.tiles_per_seg;
            seg += 1;
        }
    }
    // first element and valid length of the current tile
    __device__ __forceinline__ void span(const StreamArgs& a, long long& j0, int& len) const
    {
        const long long lo = a.base + seg * a.seg_stride;
        long long hi = lo + a.seg_len;
        if (hi > a.limit) hi = a.limit;
        const long long tt = (a.flags & F_REVERSE) ? a.tiles_per_seg - 1 - t : t;
        j0 = lo + tt * kTile;
        const long long l = hi - j0;
        len = l <= 0 ? 0 : (l > kTile ? kTile : static_cast<int>(l));
    }
};

// int8 code e of a packed word whose bytes were biased by 0x80 (wb = w ^
// 0x80808080), as a float: the byte becomes the low mantissa bits of 2^23,
// so the float is 2^23 + code + 128 exactly, and the subtraction is exact.
// Full-rate FP ops instead of integer-to-float conversions.
__device__ __forceinline__ float code_f32(uint32_t wb, int e)
{
    return __fsub_rn(__uint_as_float(__byte_perm(wb, 0x4B000000u, 0x7540u + e)), 8388736.0f);
}

// scale of rank r's block holding chunk row ch of the current tile (global)
__device__ __forceinline__ float rank_scale(const StreamArgs& a, int r, long long seg, long long t, int ch)
{
    return __ldg(a.q_rank_scales + (seg * a.q_blocks_per_shard + t * kChunksPerThread + ch) * a.q_rank_scale_stride +
                 r);
}

// Which elements of a tile a consumer thread takes: chunk ch of thread tid
// covers the tile's elements [4q, 4q + 4), q = chunk_of(ch, tid).  By default
// the chunks form rows (row ch = all consumers, one 2048-element block per
// row).  With the fused int8 gather (kHalves) each half of the consumers
// takes one 2048-element block (warps 0-7 the first, 8-15 the second), so the
// block's absmax is a barrier of 8 warps instead of 16.
template <bool kHalves>
__device__ __forceinline__ int chunk_of(int ch, int tid)
{
    if constexpr (kHalves) {
        constexpr int kHalf = kConsumers / 2;
        return (tid / kHalf) * (kQuantBlock / kChunk) + ch * kHalf + (tid % kHalf);
    } else {
        return ch * kConsumers + tid;
    }
}

// the 2048-element block (0 or 1) of the tile that chunk ch of thread tid lies in
template <bool kHalves>
__device__ __forceinline__ int block_of(int ch, int tid)
{
    return kHalves ? tid / (kConsumers / 2) : ch;
}

// rank-ordered add of one rank's dequantized codes: acc += fl(code * scale).
// kDecode 0: scalar; 1: the codes decoded (an exact subtraction) and scaled
// on register pairs, then added one by one; 2: all three on register pairs.
// Each is the same rounding sequence, one IEEE operation per step (checked
// bit for bit against the oracle); the pair forms issue fewer instructions.
template <int kDecode>
__device__ __forceinline__ void add_codes(float (&acc)[4], uint32_t w, float s)
{
    const uint32_t wb = w ^ 0x80808080u;
    if constexpr (kDecode == 0) {
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] = __fadd_rn(acc[e], __fmul_rn(code_f32(wb, e), s));
    } else {
        const f32x2 bias = pack2(8388736.0f, 8388736.0f), sc = pack2(s, s);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const f32x2 x = pack2(__uint_as_float(__byte_perm(wb, 0x4B000000u, 0x7540u + 2 * h)),
                                  __uint_as_float(__byte_perm(wb, 0x4B000000u, 0x7541u + 2 * h)));
            const f32x2 prod = mul2(sub2(x, bias), sc);
            if constexpr (kDecode == 1) {
                float p0, p1;
                unpack2(prod, p0, p1);
                acc[2 * h] = __fadd_rn(acc[2 * h], p0);
                acc[2 * h + 1] = __fadd_rn(acc[2 * h + 1], p1);
            } else {
                unpack2(add2(pack2(acc[2 * h], acc[2 * h + 1]), prod), acc[2 * h], acc[2 * h + 1]);
            }
        }
    }
}

template <int GT>
__device__ __forceinline__ void add_slice(float (&acc)[4], uint2 w)
{
    unsigned short h[4];
    halves(w.x, h[0], h[1]);
    halves(w.y, h[2], h[3]);
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[e] = Lp<GT>::add(acc[e], h[e]);
}

// rank slices per pipeline stage: int8 slices are half the bytes of 16-bit
// ones, so a stage takes twice as many to move the same bytes per barrier
template <int GT>
__host__ __device__ constexpr int group_ranks() { return GT == kGradQ8 ? 2 * kGroupRanks : kGroupRanks; }

// CTAs of one launch resident per SM.  The reduce pass over int8 codes is
// bound by instruction issue, not by DRAM: two CTAs per SM (56 registers a
// thread, which it needs no more than) give each scheduler twice the warps
// to pick from, and took the clipped GPT-2-small qgZ step from 0.838 to
// 0.806 ms.  Every other pass needs its 96 registers (at 56 they spill).
template <int GT, int OP>
__host__ __device__ constexpr int ctas_per_sm() { return (OP == OP_REDUCE && GT == kGradQ8) ? 2 : 1; }

// 17 warps spread over an SM's 4 sub-partitions put 5 on one of them, whose
// 16K registers then allow 96 per thread: the bound ptxas works to here (with
// one CTA per SM).
template <int GT, int PT, int OP, int FULL>
__global__ void __launch_bounds__(kThreads, ctas_per_sm<GT, OP>()) k_stream(const __grid_constant__ StreamArgs a)
{
    constexpr int kG = group_ranks<GT>();
    extern __shared__ __align__(1024) unsigned char smem[];
    Shared* sh = reinterpret_cast<Shared*>(smem);
    unsigned char* ring = smem + kStageOffset;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    constexpr bool quant = OP == OP_QFUSED || OP == OP_QADAM;
    // the int8 gather over int8 rank streams takes one quantization block per
    // half of the consumers (an 8-warp absmax barrier): 7% faster at N_d = 8
    // than one block per chunk row; with 16-bit rank streams the chunk rows
    // (a 16-warp barrier) measured 1-8% faster, and stay
    constexpr bool kHalves = quant && GT == kGradQ8;
    // int8 rank streams: the codes decoded and scaled on register pairs (the
    // reduce pass 4%, the int8-gather step 11% faster at N_d = 8), except in
    // the fused step with a partly filled rank group, which measured 2% faster
    // with the scalar form
    constexpr int kDecode = (OP == OP_FUSED && FULL == kPartial) ? 0 : 1;

    // The ring's barriers first, so that the producer can start copying while
    // the consumers read the step scalars (their latency then overlaps the
    // first copies).  Only a guarded pass reads its flag before producing.
    if (tid == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&sh->full[s], 1);
            mbar_init(&sh->empty[s], kConsumerWarps);
            sh->issued_parity[s] = -1;
        }
        sh->abort = 0;
        sh->skip = (a.flags & F_GUARD) ? (a.sc->nonfinite != 0) : 0;
        fence_barrier_init();
    }
    __syncthreads();
    // a flagged loss-scaling step writes nothing (uniform over the CTA)
    const bool skip = sh->skip != 0;

    const int n_groups = a.n_ranks > 0 ? (a.n_ranks + kG - 1) / kG : 1;
    const int rank_slots = a.n_ranks < kG ? a.n_ranks : kG;
    constexpr uint32_t kEB = (GT == kGradQ8) ? 1u : 2u;   // bytes per rank element
    // int8 ranks: the group's block scales (2 blocks x 8 ranks) follow the rank slices
    constexpr uint32_t kScaleBytes = (GT == kGradQ8) ? kChunksPerThread * kG * 4u : 0u;
    const uint32_t scale_off = static_cast<uint32_t>(rank_slots) * kTile * kEB;
    const uint32_t side_off = scale_off + kScaleBytes;

    bool nonfinite = false;
    f32x2 sq_hi = pack2(0.0f, 0.0f), sq_lo = pack2(0.0f, 0.0f);

    if (skip) {
        // nothing to do but record the norm (CTA 0); fall through to the end
        // (the epilogue still runs)
        if (warp == 0 && blockIdx.x == 0 && (a.flags & F_FINALIZE)) step_constants(a, sh, lane);
    } else if (warp == kConsumerWarps) {
        // ------------------------------------------------------- producer
        if (lane == 0 && !(a.flags & F_DEBUG_STARVE)) {
            int s = 0;
            uint32_t ph = 0;
            TileCursor cur;
            for (cur.start(a); cur.valid(a) && !*reinterpret_cast<volatile int*>(&sh->abort); cur.next(a)) {
                long long j0;
                int len;
                cur.span(a, j0, len);
                if (len != kTile || !a.tma_ok) continue;
                // int8 ranks: the row of scales of the tile's first block
                const float* srow = (GT == kGradQ8)
                                        ? a.q_rank_scales + (cur.seg * a.q_blocks_per_shard + cur.t * kChunksPerThread) *
                                                                a.q_rank_scale_stride
                                        : nullptr;
                for (int g = 0; g < n_groups; ++g) {
                    if (!mbar_wait_bounded(&sh->empty[s], ph ^ 1u, &sh->abort, a.timeout_ns)) {
                        atomicExch(&sh->abort, 1);
                        break;
                    }
                    const int r0 = g * kG;
                    const int nr = a.n_ranks - r0 < kG ? a.n_ranks - r0 : kG;
                    const bool last = g == n_groups - 1;
                    const uint32_t rank_bytes = kTile * kEB;
                    // int8 ranks: this group's scales of the tile's two blocks, rounded up to 4 ranks
                    // (the wire layout pads ranks to a multiple of 4, so the copy stays in bounds)
                    const uint32_t nsc = (GT == kGradQ8) ? static_cast<uint32_t>((nr + 3) / 4 * 4) : 0u;
                    const uint32_t bytes = (nr > 0 ? nr : 0) * rank_bytes + (last ? a.n_side_tma * kTile * 4u : 0u) +
                                           kChunksPerThread * nsc * 4u;
                    unsigned char* st = ring + static_cast<size_t>(s) * a.stage_bytes;
                    mbar_arrive_expect_tx(&sh->full[s], bytes);
                    if constexpr (GT == kGradQ8) {
                        for (int ch = 0; ch < kChunksPerThread; ++ch)
                            bulk_load(st + scale_off + ch * kG * 4u, srow + ch * a.q_rank_scale_stride + r0,
                                      nsc * 4u, &sh->full[s]);
                    }
                    for (int k = 0; k < nr; ++k)
                        bulk_load(st + k * rank_bytes, static_cast<const unsigned char*>(a.rank[r0 + k]) + j0 * kEB,
                                  rank_bytes, &sh->full[s]);
                    if (last)
                        for (int k = 0; k < a.n_side_tma; ++k)
                            bulk_load(st + side_off + k * kTile * 4u, a.side[k] + j0, kTile * 4u, &sh->full[s]);
                    sh->issued_parity[s] = static_cast<int>(ph);
                    if (++s == a.stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------- consumers
        int s = 0;
        uint32_t ph = 0;
        bool alive = true;
        int qiter = 0;  // quantizer barriers passed: picks the reduction buffer
        // the step constants: warp 0 computes them while the producer issues
        // the first copies; then the consumers (only) wait for them
        if (warp == 0) step_constants(a, sh, lane);
        named_bar_sync(3, kConsumers);
        // constants in registers: a reference into shared memory would be
        // re-read for every element (the stores in the loop may alias it)
        const StepConsts c = sh->c;
        // the reduce pass over int8 codes (the clipped quantized exchange) has
        // no side stream, carry or raw sum, no non-finite test, and always sums
        // squares: its flags are constants, and the tests of the other
        // passes' flags drop out of its loop
        constexpr bool kCodesReduce = OP == OP_REDUCE && GT == kGradQ8;
        constexpr int kSides = kCodesReduce ? 0 : kMaxSide;   // side streams this pass can have
        const bool detect = !kCodesReduce && (a.flags & F_DETECT) != 0;   // recorded only under loss scaling
        const bool want_sq = kCodesReduce || (a.flags & F_SQNORM) != 0;
        const bool carry = !kCodesReduce && (a.flags & F_CARRY) != 0;
        const bool raw = !kCodesReduce && (a.flags & F_RAW) != 0;
        constexpr int kCarry = (OP == OP_REDUCE) ? 0 : 3;   // side slot of the carry stream
        TileCursor cur;
        for (cur.start(a); cur.valid(a); cur.next(a)) {
            long long j0;
            int len;
            cur.span(a, j0, len);
            if (len <= 0) {
                if (quant && tid == 0) {
                    for (int ch = 0; ch < kChunksPerThread; ++ch) {
                        const long long blk = cur.t * kChunksPerThread + ch;
                        if (blk < a.q_blocks_per_shard) a.q_scales[cur.seg * a.q_blocks_per_shard + blk] = 0.0f;
                    }
                }
                continue;
            }
            const bool fast = len == kTile && a.tma_ok;
            float acc[kChunksPerThread][4];
            float sv[kChunksPerThread][kMaxSide][4];
#pragma unroll
            for (int ch = 0; ch < kChunksPerThread; ++ch)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc[ch][e] = 0.0f;
#pragma unroll
                    for (int k = 0; k < kSides; ++k) sv[ch][k][e] = 0.0f;
                }

            if (fast) {
                // side streams not staged (state in host memory): 16-byte loads issued
                // now, before the wait for the gradient stage, so their latency overlaps it
                if (kSides > 0 && a.n_side_tma < a.n_side && alive) {
#pragma unroll
                    for (int ch = 0; ch < kChunksPerThread; ++ch) {
                        const long long jc = j0 + chunk_of<kHalves>(ch, tid) * 4;
#pragma unroll
                        for (int k = 0; k < kMaxSide; ++k) {
                            if (k >= a.n_side_tma && k < a.n_side) {
                                const float4 f = *reinterpret_cast<const float4*>(a.side[k] + jc);
                                sv[ch][k][0] = f.x;
                                sv[ch][k][1] = f.y;
                                sv[ch][k][2] = f.z;
                                sv[ch][k][3] = f.w;
                            }
                        }
                    }
                }
                for (int g = 0; g < n_groups; ++g) {
                    if (alive && !mbar_wait_bounded(&sh->full[s], ph, &sh->abort, a.timeout_ns)) {
                        alive = false;
                        atomicExch(&sh->abort, 1);
                    }
                    if (alive) {
                        const unsigned char* st = ring + static_cast<size_t>(s) * a.stage_bytes;
                        const int r0 = g * kG;
                        const int nr = a.n_ranks - r0 < kG ? a.n_ranks - r0 : kG;
                        // Every group full (N_d a multiple of the group size): a loop
                        // of constant trip count, constant shared-memory offsets and no
                        // loop tests; otherwise one bounded at run time.  How far it is
                        // unrolled was measured per case (int8 ranks: fully when a tile
                        // has several groups, by 8 when it has one).
                        if constexpr (GT == kGradQ8) {
                            // scales of this group's ranks arrived with the stage (broadcast reads)
                            const float* ssc = reinterpret_cast<const float*>(st + scale_off);
#pragma unroll
                            for (int ch = 0; ch < kChunksPerThread; ++ch) {
                                const int q = chunk_of<kHalves>(ch, tid);
                                const int qb = block_of<kHalves>(ch, tid);   // the chunk's block: its scales
                                if constexpr (FULL == kFullMulti) {
                                    const uint32_t* cw = reinterpret_cast<const uint32_t*>(st) + q;
#pragma unroll
                                    for (int k = 0; k < kG; ++k) add_codes<kDecode>(acc[ch], cw[k * (kTile / 4)], ssc[qb * kG + k]);
                                } else if constexpr (FULL == kFullOne || FULL == kFullHalf) {
                                    // four ranks' scales per 16-byte shared load
                                    const uint32_t* cw = reinterpret_cast<const uint32_t*>(st) + q;
                                    const float4* s4 = reinterpret_cast<const float4*>(ssc + qb * kG);
                                    auto four = [&](int k4) {
                                        const float4 sc4 = s4[k4];
                                        add_codes<kDecode>(acc[ch], cw[(4 * k4 + 0) * (kTile / 4)], sc4.x);
                                        add_codes<kDecode>(acc[ch], cw[(4 * k4 + 1) * (kTile / 4)], sc4.y);
                                        add_codes<kDecode>(acc[ch], cw[(4 * k4 + 2) * (kTile / 4)], sc4.z);
                                        add_codes<kDecode>(acc[ch], cw[(4 * k4 + 3) * (kTile / 4)], sc4.w);
                                    };
                                    if constexpr (FULL == kFullOne) {
#pragma unroll 2
                                        for (int k4 = 0; k4 < kG / 4; ++k4) four(k4);
                                    } else {
#pragma unroll
                                        for (int k4 = 0; k4 < kG / 8; ++k4) four(k4);
                                    }
                                } else {
#pragma unroll 4
                                    for (int k = 0; k < nr; ++k) {
                                        const uint32_t w = reinterpret_cast<const uint32_t*>(st + k * kTile)[q];
                                        add_codes<kDecode>(acc[ch], w, ssc[qb * kG + k]);
                                    }
                                }
                            }
                        } else {
#pragma unroll
                            for (int ch = 0; ch < kChunksPerThread; ++ch) {
                                const int q = chunk_of<kHalves>(ch, tid);  // chunk index within the tile
                                const uint2* rw = reinterpret_cast<const uint2*>(st) + q;
                                if constexpr (FULL != kPartial && OP == OP_QFUSED) {
                                    // the int8-gather step measured fastest in this form
                                    if (nr == kG) {
#pragma unroll
                                        for (int k = 0; k < kG; ++k) add_slice<GT>(acc[ch], rw[k * (kTile / 4)]);
                                    } else {
#pragma unroll 8
                                        for (int k = 0; k < nr; ++k) add_slice<GT>(acc[ch], rw[k * (kTile / 4)]);
                                    }
                                } else if constexpr (FULL != kPartial) {
#pragma unroll
                                    for (int k = 0; k < kG; ++k) add_slice<GT>(acc[ch], rw[k * (kTile / 4)]);
                                } else {
#pragma unroll 8
                                    for (int k = 0; k < nr; ++k) add_slice<GT>(acc[ch], rw[k * (kTile / 4)]);
                                }
                            }
                        }
                        if (g == n_groups - 1) {
#pragma unroll
                            for (int ch = 0; ch < kChunksPerThread; ++ch) {
                                const int q = chunk_of<kHalves>(ch, tid);
#pragma unroll
                                for (int k = 0; k < kSides; ++k) {
                                    if (k < a.n_side_tma) {
                                        const float4 f = reinterpret_cast<const float4*>(
                                            st + side_off + k * kTile * 4)[q];
                                        sv[ch][k][0] = f.x;
                                        sv[ch][k][1] = f.y;
                                        sv[ch][k][2] = f.z;
                                        sv[ch][k][3] = f.w;
                                    }
                                }
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0 && alive) mbar_arrive(&sh->empty[s]);
                    if (++s == a.stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            } else if (alive) {
                // plain-load path: per element, bounds-checked against len
#pragma unroll
                for (int ch = 0; ch < kChunksPerThread; ++ch) {
                    const int q = chunk_of<kHalves>(ch, tid);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int idx = q * 4 + e;
                        if (idx < len) {
                            const long long j = j0 + idx;
                            for (int r = 0; r < a.n_ranks; ++r) {
                                if constexpr (GT == kGradQ8) {
                                    const float code = static_cast<float>(static_cast<const signed char*>(a.rank[r])[j]);
                                    acc[ch][e] = __fadd_rn(acc[ch][e], __fmul_rn(code, rank_scale(a, r, cur.seg, cur.t,
                                                                                                  block_of<kHalves>(ch, tid))));
                                } else {
                                    acc[ch][e] = Lp<GT>::add(acc[ch][e], static_cast<const uint16_t*>(a.rank[r])[j]);
                                }
                            }
#pragma unroll
                            for (int k = 0; k < kSides; ++k)
                                if (k < a.n_side) sv[ch][k][e] = a.side[k][j];
                        }
                    }
                }
            }

            // ------------------------------------------------ apply the op
            float xq[kChunksPerThread][4];  // 16-bit results kept for the quantizer
#pragma unroll
            for (int ch = 0; ch < kChunksPerThread; ++ch) {
                const int q = chunk_of<kHalves>(ch, tid);
                const long long jc = j0 + q * 4;
                int cnt = len - q * 4;
                cnt = cnt < 0 ? 0 : (cnt > 4 ? 4 : cnt);
                if (OP == OP_REDUCE) {
                    // uniform tests once per chunk; the squares are still added in element order
                    float gv[4], sum[4];
                    if (carry) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) sum[e] = __fadd_rn(sv[ch][kCarry][e], acc[ch][e]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e) sum[e] = acc[ch][e];
                    }
                    if (raw) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) gv[e] = sum[e];
                    } else {
                        mean_of4(c, sum, gv);
                    }
                    // elements past the tile's valid length are +0 here (nothing was
                    // added to them): finite, and their squares add nothing
                    if (detect) {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (!is_finite_f32(gv[e])) nonfinite = true;
                    }
                    if (want_sq) {
#pragma unroll
                        for (int e = 0; e < 4; e += 2) sq_accumulate2(gv[e], gv[e + 1], sq_hi, sq_lo);
                    }
                    if (alive && a.out_f32[0] != nullptr) {
                        if (fast) {
                            *reinterpret_cast<float4*>(a.out_f32[0] + jc) = make_float4(gv[0], gv[1], gv[2], gv[3]);
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                if (e < cnt) a.out_f32[0][jc + e] = gv[e];
                        }
                    }
                } else {
                    // OP_FUSED / OP_QFUSED: side = {master, m, v[, carry]};
                    // OP_ADAM / OP_QADAM: side = {g, master, m, v}
                    constexpr int P = (OP == OP_ADAM || OP == OP_QADAM) ? 1 : 0;
                    // uniform tests (divisor form, carry, detection, clip, decay)
                    // made once per chunk, not once per element -- except in the
                    // int8-gather step and with int8 ranks, whose register budget
                    // measured faster with the per-element form
                    float pv[4], mv[4], vv[4], gv[4];
                    uint16_t lp[4];
                    if constexpr (quant || GT == kGradQ8) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float g;
                            if constexpr (OP == OP_QADAM)
                                g = sv[ch][0][e];
                            else
                                g = mean_of(c, carry ? __fadd_rn(sv[ch][kCarry][e], acc[ch][e]) : acc[ch][e]);
                            if (detect && e < cnt && !is_finite_f32(g)) nonfinite = true;
                            if (c.clip) g = __fmul_rn(g, c.coef);
                            pv[e] = sv[ch][P + 0][e];
                            mv[e] = sv[ch][P + 1][e];
                            vv[e] = sv[ch][P + 2][e];
                            adam_elem(c, g, pv[e], mv[e], vv[e]);
                            lp[e] = Lp<PT>::narrow(pv[e]);
                            xq[ch][e] = Lp<PT>::widen(lp[e]);
                        }
                    } else {
                    if constexpr (OP == OP_ADAM) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) gv[e] = sv[ch][0][e];
                    } else {
                        float sum[4];
                        if (carry) {
#pragma unroll
                            for (int e = 0; e < 4; ++e) sum[e] = __fadd_rn(sv[ch][kCarry][e], acc[ch][e]);
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e) sum[e] = acc[ch][e];
                        }
                        mean_of4(c, sum, gv);
                    }
                    if (detect) {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (e < cnt && !is_finite_f32(gv[e])) nonfinite = true;
                    }
                    if (c.clip) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) gv[e] = __fmul_rn(gv[e], c.coef);
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        pv[e] = sv[ch][P + 0][e];
                        mv[e] = sv[ch][P + 1][e];
                        vv[e] = sv[ch][P + 2][e];
                    }
                    adam_elem4(c, gv, pv, mv, vv);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        lp[e] = Lp<PT>::narrow(pv[e]);
                        xq[ch][e] = Lp<PT>::widen(lp[e]);
                    }
                    }
                    if (alive) {
                        if (fast) {
                            *reinterpret_cast<float4*>(a.out_f32[0] + jc) = make_float4(pv[0], pv[1], pv[2], pv[3]);
                            *reinterpret_cast<float4*>(a.out_f32[1] + jc) = make_float4(mv[0], mv[1], mv[2], mv[3]);
                            *reinterpret_cast<float4*>(a.out_f32[2] + jc) = make_float4(vv[0], vv[1], vv[2], vv[3]);
                            if (!quant && a.out_lp != nullptr) {
                                uint2 w;
                                w.x = static_cast<uint32_t>(lp[0]) | (static_cast<uint32_t>(lp[1]) << 16);
                                w.y = static_cast<uint32_t>(lp[2]) | (static_cast<uint32_t>(lp[3]) << 16);
                                *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out_lp) + jc) = w;
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                if (e < cnt) {
                                    a.out_f32[0][jc + e] = pv[e];
                                    a.out_f32[1][jc + e] = mv[e];
                                    a.out_f32[2][jc + e] = vv[e];
                                    if (!quant && a.out_lp != nullptr) static_cast<uint16_t*>(a.out_lp)[jc + e] = lp[e];
                                }
                            }
                        }
                    }
                }
            }

            if constexpr (quant) {
                if constexpr (kHalves) {
                    // one quantization block per half of the consumers: the thread's
                    // chunks lie in block qb = tid / 256; absmax over the block's 8
                    // warps, then codes + dequantized bf16
                    constexpr int kHalf = kConsumers / 2;
                    const int qb = tid / kHalf;
                    float amax = 0.0f;
#pragma unroll
                    for (int ch = 0; ch < kChunksPerThread; ++ch)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (chunk_of<true>(ch, tid) * 4 + e < len) amax = fmaxf(amax, fabsf(xq[ch][e]));
                    amax = warp_max_f32(amax);
                    // two buffers used alternately: between two uses of one buffer every
                    // warp of the half has passed the barrier of the other, so reads are done
                    const int par = qiter & 1;
                    ++qiter;
                    if (lane == 0) sh->red_f[par][0][warp] = amax;
                    named_bar_sync(1 + qb, kHalf);
                    float m = 0.0f;
                    {
                        const float4* rv = reinterpret_cast<const float4*>(sh->red_f[par][0] + qb * (kConsumerWarps / 2));
#pragma unroll
                        for (int w = 0; w < kConsumerWarps / 8; ++w) {
                            const float4 f = rv[w];
                            m = fmaxf(m, fmaxf(fmaxf(f.x, f.y), fmaxf(f.z, f.w)));
                        }
                    }
                    const float scale = __fdiv_rn(m, 127.0f);
                    const long long blk = cur.t * kChunksPerThread + qb;   // block index within the shard
                    if (tid % kHalf == 0 && alive && blk < a.q_blocks_per_shard)
                        a.q_scales[cur.seg * a.q_blocks_per_shard + blk] = (len > qb * kQuantBlock) ? scale : 0.0f;
                    const float inv_scale = quant_reciprocal(scale);
#pragma unroll
                    for (int ch = 0; ch < kChunksPerThread; ++ch) {
                        const int q = chunk_of<true>(ch, tid);
                        const long long jc = j0 + q * 4;
                        int cnt = len - q * 4;
                        cnt = cnt < 0 ? 0 : (cnt > 4 ? 4 : cnt);
                        float cf[4];
                        const uint32_t cw = quant_code4(xq[ch], scale, inv_scale, cf);
                        const uint32_t d01 = Lp<ZERO_BF16>::narrow2(__fmul_rn(cf[0], scale), __fmul_rn(cf[1], scale));
                        const uint32_t d23 = Lp<ZERO_BF16>::narrow2(__fmul_rn(cf[2], scale), __fmul_rn(cf[3], scale));
                        const uint16_t dq[4] = {static_cast<uint16_t>(d01), static_cast<uint16_t>(d01 >> 16),
                                                static_cast<uint16_t>(d23), static_cast<uint16_t>(d23 >> 16)};
                        if (!alive) continue;
                        if (fast) {
                            *reinterpret_cast<uint32_t*>(a.q_codes + jc) = cw;
                            *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.q_gathered) + jc) = make_uint2(d01, d23);
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                if (e < cnt) {
                                    a.q_codes[jc + e] = static_cast<signed char>(static_cast<uint8_t>(cw >> (8 * e)));
                                    static_cast<uint16_t*>(a.q_gathered)[jc + e] = dq[e];
                                }
                            }
                        }
                    }
                } else {
                    // one quantization block per chunk row (all consumers x 4 elements):
                    // amax per row over the consumers, then codes + dequantized bf16
                    float amax[kChunksPerThread];
#pragma unroll
                    for (int ch = 0; ch < kChunksPerThread; ++ch) {
                        amax[ch] = 0.0f;
                        if (fast) {   // every element valid: no per-element bound test
#pragma unroll
                            for (int e = 0; e < 4; ++e) amax[ch] = fmaxf(amax[ch], fabsf(xq[ch][e]));
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                if ((ch * kConsumers + tid) * 4 + e < len) amax[ch] = fmaxf(amax[ch], fabsf(xq[ch][e]));
                        }
                        amax[ch] = warp_max_f32(amax[ch]);
                    }
                    // two buffers used alternately: between two uses of one buffer every
                    // consumer has passed the barrier of the other, so reads are done
                    const int par = qiter & 1;
                    ++qiter;
                    if (lane == 0) {
#pragma unroll
                        for (int ch = 0; ch < kChunksPerThread; ++ch) sh->red_f[par][ch][warp] = amax[ch];
                    }
                    named_bar_sync(1, kConsumers);
#pragma unroll
                    for (int ch = 0; ch < kChunksPerThread; ++ch) {
                        float m = 0.0f;
                        const float4* rv = reinterpret_cast<const float4*>(sh->red_f[par][ch]);
#pragma unroll
                        for (int w = 0; w < kConsumerWarps / 4; ++w) {
                            const float4 f = rv[w];
                            m = fmaxf(m, fmaxf(fmaxf(f.x, f.y), fmaxf(f.z, f.w)));
                        }
                        const float scale = __fdiv_rn(m, 127.0f);
                        const long long blk = cur.t * kChunksPerThread + ch;   // block index within the shard
                        if (tid == 0 && alive && blk < a.q_blocks_per_shard)
                            a.q_scales[cur.seg * a.q_blocks_per_shard + blk] = (len > ch * kQuantBlock) ? scale : 0.0f;
                        const float inv_scale = quant_reciprocal(scale);
                        const int q = ch * kConsumers + tid;
                        const long long jc = j0 + q * 4;
                        int cnt = len - q * 4;
                        cnt = cnt < 0 ? 0 : (cnt > 4 ? 4 : cnt);
                        float cf[4];
                        const uint32_t cw = quant_code4(xq[ch], scale, inv_scale, cf);
                        // the dequantized products on register pairs (they feed the
                        // bf16 conversion, nothing to contract with)
                        float q0, q1, q2, q3;
                        unpack2(mul2(pack2(cf[0], cf[1]), pack2(scale, scale)), q0, q1);
                        unpack2(mul2(pack2(cf[2], cf[3]), pack2(scale, scale)), q2, q3);
                        const uint32_t d01 = Lp<ZERO_BF16>::narrow2(q0, q1);
                        const uint32_t d23 = Lp<ZERO_BF16>::narrow2(q2, q3);
                        const uint16_t dq[4] = {static_cast<uint16_t>(d01), static_cast<uint16_t>(d01 >> 16),
                                                static_cast<uint16_t>(d23), static_cast<uint16_t>(d23 >> 16)};
                        if (!alive) continue;
                        if (fast) {
                            *reinterpret_cast<uint32_t*>(a.q_codes + jc) = cw;
                            *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.q_gathered) + jc) = make_uint2(d01, d23);
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                if (e < cnt) {
                                    a.q_codes[jc + e] = static_cast<signed char>(static_cast<uint8_t>(cw >> (8 * e)));
                                    static_cast<uint16_t*>(a.q_gathered)[jc + e] = dq[e];
                                }
                            }
                        }
                    }
                }
            }
        }
    }

    // ------------------------------------------------------------ CTA end
    const int any_nonfinite = __syncthreads_or(nonfinite ? 1 : 0);
    if (tid == 0 && any_nonfinite && (a.flags & F_DETECT)) atomicOr(&a.sc->nonfinite, 1);
    if (OP == OP_REDUCE && (a.flags & F_SQNORM)) {
        float h0, h1, l0, l1;
        unpack2(sq_hi, h0, h1);
        unpack2(sq_lo, l0, l1);
        double part = warp < kConsumerWarps ? __dadd_rn(__dadd_rn(static_cast<double>(h0), static_cast<double>(l0)),
                                                        __dadd_rn(static_cast<double>(h1), static_cast<double>(l1))) : 0.0;
        part = warp_sum_f64(part);
        if (lane == 0 && warp < kConsumerWarps) sh->red_d[warp] = part;
        __syncthreads();
        if (tid == 0) {
            double tot = 0.0;
            for (int w = 0; w < kConsumerWarps; ++w) tot = __dadd_rn(tot, sh->red_d[w]);
            a.partials[blockIdx.x] = tot;
        }
    }
    if (tid == 0 && sh->abort) {
        // a wait ran out: let every copy already issued land before the CTA
        // gives its shared memory back, then report
        for (int s = 0; s < a.stages; ++s)
            if (sh->issued_parity[s] >= 0)
                mbar_wait_bounded(&sh->full[s], static_cast<uint32_t>(sh->issued_parity[s]), nullptr, a.timeout_ns);
        if (a.sc != nullptr) atomicOr(&a.sc->status, ZERO_DEV_TIMEOUT);
    }
    if (a.flags & F_EPILOGUE) {
        // the last CTA to finish commits the step scalars: every CTA read them
        // in its prologue before taking its ticket (no CTA waits for another)
        if (tid == 0) {
            __threadfence();
            const unsigned done = atomicAdd(&a.sc->ctas_done, 1u);
            if (done == gridDim.x - 1) {
                __threadfence();
                commit_scalars(a.hp, a.sc);
                a.sc->ctas_done = 0u;
            }
        }
    }
}

// ---------------------------------------------------------------- launching
namespace {

struct DevInfo {
    int sms = 0;
    int smem_optin = 0;
    int smem_per_sm = 0;
    int smem_reserved = 0;   // per CTA, by the runtime
};

DevInfo device_info(int dev)
{
    static DevInfo cache[64];
    static int ready[64];
    if (dev < 0 || dev >= 64) return DevInfo{};
    if (!__atomic_load_n(&ready[dev], __ATOMIC_ACQUIRE)) {
        DevInfo d;
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        cudaDeviceGetAttribute(&d.smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
        cache[dev] = d;
        __atomic_store_n(&ready[dev], 1, __ATOMIC_RELEASE);
    }
    return cache[dev];
}

template <int GT, int PT, int OP, int FULL>
cudaError_t launch_one_k(StreamArgs& a, cudaStream_t st)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const DevInfo di = device_info(dev);
    if (di.sms <= 0) return cudaErrorInvalidDevice;
    // stage size: rank slots + fp32 side streams of one tile
    constexpr int kG = group_ranks<GT>();
    const int slots = a.n_ranks < kG ? a.n_ranks : kG;
    const int eb = (GT == kGradQ8) ? 1 : 2;
    const int scale_bytes = (GT == kGradQ8) ? kChunksPerThread * kG * 4 : 0;
    a.stage_bytes = static_cast<unsigned>(slots * kTile * eb + scale_bytes + a.n_side_tma * kTile * 4);
    int stages = (di.smem_optin - kStageOffset) / static_cast<int>(a.stage_bytes);
    // the deeper ring where a side stream is not staged (state in host memory,
    // the fused step over 16 or more int8 ranks, an accumulation carry: with
    // the carry the GPT-2-small 4-micro-batch step measured the same either way)
    const int ring = ((a.flags & F_HOST_STATE) || a.n_side_tma < a.n_side) ? kMaxStages : kRingStages;
    if (stages > ring) stages = ring;
    if (stages < 2) return cudaErrorInvalidConfiguration;
    a.stages = stages;
    const size_t smem = kStageOffset + static_cast<size_t>(stages) * a.stage_bytes;
    static int attr_done[64];
    if (dev < 64 && !__atomic_load_n(&attr_done[dev], __ATOMIC_ACQUIRE)) {
        err = cudaFuncSetAttribute(k_stream<GT, PT, OP, FULL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   di.smem_optin);
        if (err != cudaSuccess) return err;
        __atomic_store_n(&attr_done[dev], 1, __ATOMIC_RELEASE);
    }
    const long long ntiles = a.tiles_per_seg * a.n_seg;
    // two CTAs per SM where the kernel is built for it and both rings fit in
    // the SM's shared memory (int8 codes of up to 13 ranks with 228 KB per
    // SM); else one
    long long per_sm = ctas_per_sm<GT, OP>();
    if (per_sm > 1 && per_sm * (static_cast<long long>(smem) + di.smem_reserved) > di.smem_per_sm) per_sm = 1;
    const long long resident = per_sm * di.sms;
    long long grid = ntiles < resident ? ntiles : resident;
    // The Adam pass and the 16-bit fused step with one rank group and its state
    // staged ran 3-8% faster on 27/32 of the SMs (128 of 152) than on all of
    // them (measured from 100 to 152 CTAs: a step between 140 and 132); fewer
    // CTAs interleave fewer streams in DRAM.  The int8-gather step, int8 ranks,
    // several rank groups, an accumulation carry and host-memory state
    // measured faster with every SM.
    if constexpr ((OP == OP_FUSED || OP == OP_ADAM) && GT != kGradQ8) {
        if (a.n_ranks <= kGroupRanks && a.n_side_tma == a.n_side && !(a.flags & F_HOST_STATE)) {
            const long long cap = (static_cast<long long>(di.sms) * 27) / 32;
            if (grid > cap) grid = cap;
        }
    }
    if (grid > kMaxPartials) grid = kMaxPartials;
    if (grid <= 0) return cudaSuccess;
    a.grid = static_cast<int>(grid);
    count_launch();
    k_stream<GT, PT, OP, FULL><<<static_cast<unsigned>(grid), kThreads, smem, st>>>(a);
    return cudaGetLastError();
}

// picks the rank-loop shape from the launch's rank count
template <int GT, int PT, int OP>
cudaError_t launch_one(StreamArgs& a, cudaStream_t st)
{
    constexpr int kG = group_ranks<GT>();
    if constexpr (OP == OP_ADAM || OP == OP_QADAM) {
        return launch_one_k<GT, PT, OP, kPartial>(a, st);
    } else {
        // eight int8 ranks: the reduce pass measured 3% faster with the loop of
        // constant trip count, the fused step 3% slower
        if constexpr (GT == kGradQ8 && OP == OP_REDUCE) {
            if (a.n_ranks == kG / 2) return launch_one_k<GT, PT, OP, kFullHalf>(a, st);
        }
        if (a.n_ranks <= 0 || a.n_ranks % kG != 0) return launch_one_k<GT, PT, OP, kPartial>(a, st);
        if constexpr (GT == kGradQ8) {
            if (a.n_ranks > kG) return launch_one_k<GT, PT, OP, kFullMulti>(a, st);
        }
        return launch_one_k<GT, PT, OP, kFullOne>(a, st);
    }
}

}  // namespace

cudaError_t launch_stream(int op, int grad_dtype, int param_dtype, StreamArgs& a, cudaStream_t st)
{
    const bool gb = grad_dtype == ZERO_BF16, pb = param_dtype == ZERO_BF16;
    if (grad_dtype == kGradQ8) {   // int8 ranks: the fused step (plain or int8 gather) and the reduce pass
        if (op == OP_REDUCE) return launch_one<kGradQ8, ZERO_BF16, OP_REDUCE>(a, st);
        if (op == OP_QFUSED) return pb ? launch_one<kGradQ8, ZERO_BF16, OP_QFUSED>(a, st) : cudaErrorInvalidValue;
        if (op != OP_FUSED) return cudaErrorInvalidValue;
        return pb ? launch_one<kGradQ8, ZERO_BF16, OP_FUSED>(a, st) : launch_one<kGradQ8, ZERO_FP16, OP_FUSED>(a, st);
    }
    switch (op) {
    case OP_FUSED:
        if (gb) return pb ? launch_one<ZERO_BF16, ZERO_BF16, OP_FUSED>(a, st) : launch_one<ZERO_BF16, ZERO_FP16, OP_FUSED>(a, st);
        return pb ? launch_one<ZERO_FP16, ZERO_BF16, OP_FUSED>(a, st) : launch_one<ZERO_FP16, ZERO_FP16, OP_FUSED>(a, st);
    case OP_REDUCE:
        return gb ? launch_one<ZERO_BF16, ZERO_BF16, OP_REDUCE>(a, st) : launch_one<ZERO_FP16, ZERO_BF16, OP_REDUCE>(a, st);
    case OP_ADAM:
        return pb ? launch_one<ZERO_BF16, ZERO_BF16, OP_ADAM>(a, st) : launch_one<ZERO_BF16, ZERO_FP16, OP_ADAM>(a, st);
    case OP_QADAM:    // the int8 gather reads bf16 parameters only
        return pb ? launch_one<ZERO_BF16, ZERO_BF16, OP_QADAM>(a, st) : cudaErrorInvalidValue;
    case OP_QFUSED:   // the int8 gather reads bf16 parameters only
        if (!pb) return cudaErrorInvalidValue;
        return gb ? launch_one<ZERO_BF16, ZERO_BF16, OP_QFUSED>(a, st) : launch_one<ZERO_FP16, ZERO_BF16, OP_QFUSED>(a, st);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace zk
