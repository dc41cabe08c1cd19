"""GPU parity: every entry point of libzero.so against the CPU oracle on the
same seeded bytes, at sizes the oracle finishes in seconds that span many
4096-element tiles plus ragged tails.

Bars: the reduce, Adam and cast use the oracle's IEEE operation order, so
master/m/v and the 16-bit parameters are compared bit for bit (which implies
the stated tolerance, relative 1e-6 and 1 ulp).  With clipping the global norm
is summed in another order on the GPU, so the coefficient may differ by an
ulp: those cases are held to the tolerance.  Layout, padding, skip decisions,
int8 codes and scales are compared exactly."""
import math

import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_02_gb300 as z
from gpu_helpers import ORACLE_DT, TORCH_DT, Job, oracle_hp, u16, u32
from zero_optimizer_step_02_gb300 import synth

pytestmark = pytest.mark.gpu

SHAPES = [  # (n_d, psi, pad)
    (1, 1, 1), (1, 5000, 8), (2, 2047, 1), (3, 40_000, 8), (4, 1_000_003, 8), (4, 1_000_003, 1),
    (5, 3, 64), (8, 123_457, 8), (16, 70_001, 64), (64, 100_000, 8), (64, 63, 1),
]


# ---------------------------------------------------------------- fused step
@pytest.mark.parametrize("n_d,psi,pad", SHAPES)
@pytest.mark.parametrize("stage", [1, 2, 3])
def test_fused_step_bit_exact(n_d, psi, pad, stage):
    job = Job(psi, n_d, stage=stage, pad=pad, hp=z.hparams(lr=1e-3), seed=psi + n_d)
    for step in range(1, 4):
        job.new_grads(step)
        job.gpu_step()
        job.oracle_step()
        job.assert_bit_exact()
    assert job.scalars().t == 3


def _small_limit():
    # a plain step below two 4096-element tiles per SM takes the small-problem
    # kernel (one thread per 4 elements, no staging); at and above, the engine
    return 2 * torch.cuda.get_device_properties(0).multi_processor_count * 4096


@pytest.mark.parametrize("offset", [-3, -1, 0, 1])
@pytest.mark.parametrize("gdt,pdt,stage", [(z.ZERO_BF16, z.ZERO_BF16, 2), (z.ZERO_FP16, z.ZERO_FP16, 3),
                                           (z.ZERO_FP16, z.ZERO_BF16, 1)])
def test_fused_step_either_side_of_the_small_problem_limit(offset, gdt, pdt, stage):
    # the small-problem kernel and the engine give the oracle's bits alike,
    # with a ragged tail on either side of the limit
    psi = _small_limit() + offset
    job = Job(psi, 3, stage=stage, pad=1, gdt=gdt, pdt=pdt, hp=z.hparams(lr=1e-3, weight_decay=0.1), seed=7)
    for step in range(1, 3):
        job.new_grads(step, sigma=1e-2)
        job.gpu_step()
        job.oracle_step()
        job.assert_bit_exact()
    assert job.scalars().t == 2


@pytest.mark.parametrize("gdt,pdt", [(z.ZERO_FP16, z.ZERO_BF16), (z.ZERO_FP16, z.ZERO_FP16),
                                     (z.ZERO_BF16, z.ZERO_FP16)])
def test_fused_step_dtypes(gdt, pdt):
    job = Job(300_007, 8, stage=2, pad=8, gdt=gdt, pdt=pdt, hp=z.hparams(lr=1e-4, weight_decay=0.01), seed=3)
    for step in range(1, 4):
        job.new_grads(step, sigma=1e-2)
        job.gpu_step()
        job.oracle_step()
        job.assert_bit_exact()


def test_fused_step_adamw_pingpong():
    job = Job(500_000, 4, stage=2, pad=8, hp=z.hparams(lr=3e-4, beta2=0.95, weight_decay=0.1), seed=5,
              pingpong=True)
    for step in range(1, 5):
        job.new_grads(step, sigma=1e-2, heavy_tail=True)
        job.gpu_step()
        job.oracle_step()
        job.assert_bit_exact()


def test_fused_step_in_buckets_equals_one_pass():
    psi, n_d = 1_000_003, 4
    a = Job(psi, n_d, hp=z.hparams(), seed=9)
    b = Job(psi, n_d, hp=z.hparams(), seed=9, bucket=300_000)
    for step in (1, 2):
        a.new_grads(step)
        b.new_grads(step)
        a.gpu_step()
        b.gpu_step()
        b.oracle_step()
        b.assert_bit_exact()
    assert np.array_equal(u32(a.buf.master.cpu().numpy()), u32(b.buf.master.cpu().numpy()))


def test_fused_step_is_deterministic():
    outs = []
    for _ in range(2):
        job = Job(777_777, 8, hp=z.hparams(max_norm=0.5, weight_decay=0.1), seed=11)
        for step in (1, 2):
            job.new_grads(step, sigma=1e-2, heavy_tail=True)
            job.gpu_step()
        outs.append([x.copy() for x in job.gpu_state()] + [job.scalars().sqnorm])
    for x, y in zip(outs[0][:4], outs[1][:4]):
        assert np.array_equal(x.view(np.uint32) if x.dtype == np.float32 else x,
                              y.view(np.uint32) if y.dtype == np.float32 else y)
    assert outs[0][4] == outs[1][4]


# ------------------------------------------------------------------ clipping
@pytest.mark.parametrize("n_d", [2, 4, 8])   # n_d <= 4 re-reads the ranks, n_d > 4 keeps g in the workspace
@pytest.mark.parametrize("pingpong", [False, True])
def test_fused_step_with_clipping(n_d, pingpong):
    psi = 400_003
    hp = z.hparams(lr=3e-4, beta1=0.9, beta2=0.95, weight_decay=0.1, max_norm=1.0)
    job = Job(psi, n_d, hp=hp, seed=21 + n_d, pingpong=pingpong)
    for step in range(1, 5):
        job.new_grads(step, sigma=1e-2, heavy_tail=True)
        job.gpu_step()
        job.oracle_step()
        sc = job.scalars()
        # both sums within the sequential fp64 sum's error bound of each other
        assert sc.sqnorm == pytest.approx(job.ost.scalars.sqnorm, rel=2 * psi * 2.0 ** -53)
        assert np.float32(job.ost.scalars.clip_coef) < 1.0   # the clip is active in this workload
        job.settle()


# -------------------------------------------------------------- loss scaling
@pytest.mark.parametrize("pingpong", [False, True])   # in place: check pass; out of place: speculative + repair
@pytest.mark.parametrize("stage", [2, 3])
def test_fp16_overflow_skip(pingpong, stage):
    psi, n_d = 600_001, 8
    hp = z.hparams(lr=1e-4, loss_scaling=True)
    job = Job(psi, n_d, stage=stage, gdt=z.ZERO_FP16, hp=hp, seed=31, pingpong=pingpong, loss_scale=1024.0)
    for step in range(1, 7):
        scale = job.ost.scalars.loss_scale
        inf_at = synth.pick_index(31, step, n_d, psi) if step == 3 else None
        job.new_grads(step, sigma=1e-4, scale=scale, inf_at=inf_at)
        before = job.gpu_state()
        job.gpu_step()
        skipped = job.oracle_step()
        sc = job.scalars()
        assert bool(sc.overflow) == skipped == (step == 3)
        assert sc.loss_scale == job.ost.scalars.loss_scale
        assert sc.t == job.ost.scalars.t and sc.good_steps == job.ost.scalars.good_steps
        assert sc.nonfinite == 0 and sc.status == 0
        job.assert_bit_exact()
        if skipped:
            after = job.gpu_state()
            for x, y in zip(before, after):
                assert np.array_equal(x, y)
    assert job.scalars().loss_scale == 512.0 and job.scalars().t == 5


def test_fp16_overflow_with_clipping():
    psi, n_d = 200_003, 8
    hp = z.hparams(lr=1e-4, loss_scaling=True, max_norm=1e-3)
    job = Job(psi, n_d, gdt=z.ZERO_FP16, hp=hp, seed=33, loss_scale=1024.0)
    for step in range(1, 5):
        inf_at = (2, 1234) if step == 2 else None
        job.new_grads(step, sigma=1e-4, scale=job.ost.scalars.loss_scale, inf_at=inf_at)
        job.gpu_step()
        skipped = job.oracle_step()
        assert bool(job.scalars().overflow) == skipped == (step == 2)
        job.settle(skipped=skipped)


# -------------------------------------------------------------- the parts
@pytest.mark.parametrize("n_d,psi,pad", [(4, 1_000_003, 8), (3, 40_000, 1), (64, 5_000, 8), (2, 2047, 1)])
@pytest.mark.parametrize("gdt", [z.ZERO_BF16, z.ZERO_FP16])
def test_reduce_scatter_bit_exact(n_d, psi, pad, gdt):
    job = Job(psi, n_d, pad=pad, gdt=gdt, hp=z.hparams(), seed=41)
    job.new_grads(1, sigma=1e-2)
    out = torch.full((job.plan.padded,), float("nan"), device="cuda")
    z.zero_reduce_scatter(job.plan.handle, job.buf.rank_list(), job.hp, job.buf.scalars, out, job.buf.ws)
    want = oracle.reduce_scatter(job.rows, ORACLE_DT[gdt], float(n_d), job.plan.shard)
    assert np.array_equal(u32(out.cpu().numpy()), u32(want))     # padding included: +0


def test_reduce_scatter_with_loss_scale():
    psi, n_d = 100_000, 8
    hp = z.hparams(loss_scaling=True)
    job = Job(psi, n_d, gdt=z.ZERO_FP16, hp=hp, seed=42, loss_scale=1024.0)
    job.new_grads(1, sigma=1e-4, scale=1024.0)
    out = torch.zeros(job.plan.padded, device="cuda")
    z.zero_reduce_scatter(job.plan.handle, job.buf.rank_list(), hp, job.buf.scalars, out, job.buf.ws)
    want = oracle.reduce_scatter(job.rows, oracle.FP16, float(n_d) * 1024.0, job.plan.shard)
    assert np.array_equal(u32(out.cpu().numpy()), u32(want))


@pytest.mark.parametrize("from_partials", [True, False])
def test_grad_sqnorm_and_coefficient(from_partials):
    psi, n_d = 2_000_001, 8
    hp = z.hparams(max_norm=1.0)
    job = Job(psi, n_d, hp=hp, seed=43)
    job.new_grads(1, sigma=1e-2, heavy_tail=True)
    g = torch.zeros(job.plan.padded, device="cuda")
    z.zero_reduce_scatter(job.plan.handle, job.buf.rank_list(), hp, job.buf.scalars, g, job.buf.ws)
    z.zero_grad_sqnorm(job.plan.handle, None if from_partials else g, hp, job.buf.scalars, job.buf.ws)
    sc = job.scalars()
    g_or = oracle.reduce_scatter(job.rows, oracle.BF16, float(n_d), job.plan.shard)
    want = oracle.sqnorm(g_or)
    # the exactly rounded sum of the exact squares (fp32 squares are exact in
    # fp64): the GPU's compensated sum must be within 1e-13 of it, the
    # oracle's sequential fp64 sum within its own bound (n - 1) * 2^-53
    exact = math.fsum(np.square(g_or.astype(np.float64)))
    assert abs(sc.sqnorm - exact) <= 1e-13 * exact
    assert abs(want - exact) <= psi * 2.0 ** -53 * exact
    coef, applied = oracle.clip_coef(1.0, want)
    assert applied
    assert abs(int(np.float32(sc.clip_coef).view(np.int32)) - int(np.float32(coef).view(np.int32))) <= 1


@pytest.mark.parametrize("stage", [2, 3])
def test_parts_compose_to_the_fused_step(stage):
    # reduce-scatter -> Adam on the shards -> (stage 3) all-gather, through the C ABI
    psi, n_d, pad = 333_333, 4, 8
    hp = z.hparams(lr=1e-3, weight_decay=0.01)
    job = Job(psi, n_d, stage=stage, pad=pad, hp=hp, seed=44)
    g = torch.zeros(job.plan.padded, device="cuda")
    for step in (1, 2):
        job.new_grads(step)
        z.zero_reduce_scatter(job.plan.handle, job.buf.rank_list(), hp, job.buf.scalars, g, job.buf.ws)
        z.zero_adam_shard_step(job.plan.handle, hp, g, job.buf.master, job.buf.m, job.buf.v, job.buf.lp,
                               job.buf.scalars)
        job.oracle_step()
        job.assert_bit_exact()
    if stage == 3:
        S = job.plan.shard
        gathered = torch.full((psi + 64,), 0x7777, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        shards = [job.buf.lp[r * S:(r + 1) * S] for r in range(n_d)]
        z.zero_all_gather(job.plan.handle, shards, gathered, job.buf.scalars)
        got = u16(gathered)
        assert np.array_equal(got[:psi], job.o_lp_shards[:psi])
        assert np.all(got[psi:] == 0x7777)           # nothing written past psi
    assert job.scalars().t == 2


@pytest.mark.parametrize("n_d,psi,pad", [(4, 1_000_003, 8), (3, 100_000, 1), (16, 218_113, 8), (2, 7, 1),
                                         (8, 8 * 8192 * 3, 8)])
def test_all_gather_bit_exact(n_d, psi, pad):
    plan = z.Plan(psi, n_d, stage=3, shard_pad=pad)
    S = plan.shard
    rng = np.random.default_rng(psi)
    flat = rng.integers(0, 2 ** 16, size=plan.padded, dtype=np.uint16)
    dev = torch.from_numpy(flat.view(np.int16)).cuda().view(torch.bfloat16)
    gathered = torch.full((psi + 16,), 0x5555, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    sc = torch.zeros(256, dtype=torch.uint8, device="cuda")
    z.zero_scalars_init(sc)
    z.zero_all_gather(plan.handle, [dev[r * S:(r + 1) * S] for r in range(n_d)], gathered, sc)
    want = oracle.all_gather_u16([flat[r * S:(r + 1) * S] for r in range(n_d)], psi, S)
    got = u16(gathered)
    assert np.array_equal(got[:psi], want) and np.all(got[psi:] == 0x5555)
    assert z.read_scalars(sc).status == 0


# ---------------------------------------------------------- quantized gather
@pytest.mark.parametrize("n_d,psi,pad,block", [(2, 1 << 20, 8, 2048), (4, 1_000_003, 8, 2048),
                                               (3, 100_000, 1, 256), (8, 5000, 8, 32), (4, 70_000, 64, 4096)])
def test_quant_gather_bit_exact(n_d, psi, pad, block):
    plan = z.Plan(psi, n_d, stage=2, shard_pad=pad)
    S = plan.shard
    x = torch.zeros(plan.padded, dtype=torch.bfloat16)
    synth.gaussian_(x[:psi], 0.02, 51, psi)
    x[:psi:997] = 0.0
    xd = x.cuda()
    nbs = -(-S // block)
    codes = torch.full((plan.padded,), 99, dtype=torch.int8, device="cuda")
    scales = torch.full((n_d * nbs,), -1.0, device="cuda")
    gathered = torch.zeros(psi, dtype=torch.bfloat16, device="cuda")
    z.zero_quant_gather(plan.handle, xd, block, codes, scales, gathered)
    oc, osc, og = oracle.quant_gather(u16(x), n_d, psi, S, block)
    assert np.array_equal(codes.cpu().numpy()[:psi], oc[:psi])
    assert np.array_equal(u32(scales.cpu().numpy()), u32(osc))
    assert np.array_equal(u16(gathered), og)


@pytest.mark.parametrize("block", [2048, 256])
def test_quant_gather_non_finite_weights(block):
    # blocks holding a NaN weight (skipped by the absmax; its code is -127)
    # or an infinite one (scale inf: finite weights code 0, the infinite one
    # -127): codes and scales bit for bit; dequantized values bit for bit
    # where the oracle's are numbers, NaN where they are NaN (a NaN's payload
    # is not part of the result)
    n_d, psi = 2, 4 * 2048 + 100
    plan = z.Plan(psi, n_d, stage=2, shard_pad=8)
    S = plan.shard
    x = torch.zeros(plan.padded, dtype=torch.bfloat16)
    synth.gaussian_(x[:psi], 0.02, 53, psi)
    for j, val in ((5, float("nan")), (block + 7, float("inf")), (block + 9, float("nan")), (S + 3, float("-inf")),
                   (S + 2 * block + 1, float("nan"))):
        x[j] = val
    xd = x.cuda()
    nbs = -(-S // block)
    codes = torch.full((plan.padded,), 99, dtype=torch.int8, device="cuda")
    scales = torch.full((n_d * nbs,), -1.0, device="cuda")
    gathered = torch.zeros(psi, dtype=torch.bfloat16, device="cuda")
    z.zero_quant_gather(plan.handle, xd, block, codes, scales, gathered)
    oc, osc, og = oracle.quant_gather(u16(x), n_d, psi, S, block)
    assert np.array_equal(codes.cpu().numpy()[:psi], oc[:psi])
    assert np.array_equal(u32(scales.cpu().numpy()), u32(osc))
    got = u16(gathered)
    o_nan = np.isnan(oracle.bf16_to_f32(og))
    assert o_nan.any() and np.array_equal(np.isnan(oracle.bf16_to_f32(got)), o_nan)
    assert np.array_equal(got[~o_nan], og[~o_nan])


@pytest.mark.parametrize("n_d,psi,pad", [(2, 1 << 20, 8), (4, 1_000_003, 8), (16, 300_001, 8), (3, 50_001, 1)])
def test_fused_quantized_gather(n_d, psi, pad):
    hp = z.hparams(lr=1e-3)
    job = Job(psi, n_d, pad=pad, hp=hp, seed=61)
    S = job.plan.shard
    nbs = -(-S // 2048)
    codes = torch.zeros(job.plan.padded, dtype=torch.int8, device="cuda")
    scales = torch.full((n_d * nbs,), -1.0, device="cuda")
    gathered = torch.zeros(psi, dtype=torch.bfloat16, device="cuda")
    for step in (1, 2):
        job.new_grads(step)
        b = job.buf
        z.zero_step_fused_qgather(job.plan.handle, hp, b.rank_list(), b.master, b.m, b.v, b.master, b.m, b.v, 2048,
                                  codes, scales, gathered, b.scalars, b.ws)
        job.oracle_step()
        # the oracle quantizes the cast of the updated master, shard by shard
        lp_flat = np.zeros(job.plan.padded, np.uint16)
        lp_flat[:psi] = job.o_gathered
        oc, osc, og = oracle.quant_gather(lp_flat, n_d, psi, S, 2048)
        gm, gmm, gv, _ = job.gpu_state()
        assert np.array_equal(u32(gm), u32(job.ost.master)) and np.array_equal(u32(gv), u32(job.ost.v))
        assert np.array_equal(codes.cpu().numpy()[:psi], oc[:psi])
        assert np.array_equal(u32(scales.cpu().numpy()), u32(osc))
        assert np.array_equal(u16(gathered), og)


# -------------------------------------------------------- bounded waits
@pytest.mark.parametrize("kernel", [0, 1, 2])   # streaming engine, all-gather ring, gradient sender
def test_pipelined_kernel_timeout_path_reports_and_context_survives(kernel):
    # a launch whose bulk copies are never issued: every wait runs out, the
    # launch reports and returns
    sc = torch.zeros(256, dtype=torch.uint8, device="cuda")
    scratch = torch.zeros(32768, dtype=torch.uint8, device="cuda")
    z.zero_scalars_init(sc)
    z.zero_debug_stream_timeout(kernel, scratch, sc, 2_000_000)
    s = z.read_scalars(sc)
    assert s.status & z.ZERO_DEV_TIMEOUT
    assert torch.count_nonzero(scratch[:8192]).item() == 0      # the input region is never touched
    job = Job(10_000, 2, hp=z.hparams(), seed=72)
    job.new_grads(1)
    job.gpu_step()
    job.oracle_step()
    job.assert_bit_exact()


def test_quant_gather_run_out_wait_reports_and_falls_back_to_global_memory():
    # the weight gather's copies are never issued: its wait runs out, it
    # reports, then quantizes the block from global memory (the same codes,
    # scale and dequantized values as the oracle's)
    sc = torch.zeros(256, dtype=torch.uint8, device="cuda")
    scratch = torch.zeros(32768, dtype=torch.uint8, device="cuda")
    x = torch.zeros(2048, dtype=torch.bfloat16)
    synth.gaussian_(x, 0.02, 53, 0)
    x[::97] = 0.0
    scratch[:4096] = x.view(torch.uint8).cuda()
    z.zero_scalars_init(sc)
    z.zero_debug_stream_timeout(3, scratch, sc, 2_000_000)
    assert z.read_scalars(sc).status & z.ZERO_DEV_TIMEOUT
    oc, osc, og = oracle.quant_gather(u16(x), 1, 2048, 2048, 2048)
    got = scratch.cpu()
    assert np.array_equal(got[4096:6144].view(torch.int8).numpy(), oc)
    assert np.array_equal(u32(got[12288:12292].view(torch.float32).numpy()), u32(osc))
    assert np.array_equal(got[8192:12288].view(torch.int16).numpy().view(np.uint16), og)


def test_bounded_wait_reports_timeout_and_context_survives():
    sc = torch.zeros(256, dtype=torch.uint8, device="cuda")
    z.zero_scalars_init(sc)
    z.zero_debug_wait_timeout(sc, 2_000_000)      # 2 ms on a barrier nothing completes
    s = z.read_scalars(sc)
    assert s.status & z.ZERO_DEV_TIMEOUT
    # the context is still usable: a normal step runs and matches the oracle
    job = Job(10_000, 2, hp=z.hparams(), seed=71)
    job.new_grads(1)
    job.gpu_step()
    job.oracle_step()
    job.assert_bit_exact()


# ------------------------------------------------------------ edge cases
@pytest.mark.parametrize("n_d,psi", [(256, 1000), (256, 1), (7, 6), (128, 2048 * 129 + 5)])
def test_many_ranks_and_tiny_models(n_d, psi):
    job = Job(psi, n_d, pad=1, hp=z.hparams(), seed=81)
    job.new_grads(1)
    job.gpu_step()
    job.oracle_step()
    job.assert_bit_exact()


def test_padding_is_never_touched():
    psi, n_d, pad = 10_001, 4, 64
    job = Job(psi, n_d, pad=pad, hp=z.hparams(weight_decay=0.1, max_norm=0.1), seed=91)
    for step in (1, 2):
        job.new_grads(step)
        job.gpu_step()
    gm, gmm, gv, _ = job.gpu_state()
    for a in (gm, gmm, gv):
        assert not u32(a[psi:]).any()


def test_quant_codes_at_and_near_ties():
    # every block holds 127 s (so s = 2^-10 exactly) and values (k + 1/2) s,
    # which are exact ties of x / s, plus values one bf16 ulp off a tie: the
    # rounding decision must match the oracle's IEEE quotient in all of them
    n_d, block = 2, 2048
    psi = n_d * 4 * block
    plan = z.Plan(psi, n_d, stage=2, shard_pad=8)
    k = np.arange(-126, 126)
    ties = (k + 0.5) * 2.0 ** -10
    vals = np.concatenate([ties, np.nextafter(ties.astype(np.float32), np.float32(np.inf)),
                           np.nextafter(ties.astype(np.float32), np.float32(-np.inf))])
    rng = np.random.default_rng(3)
    x = rng.choice(vals, size=psi).astype(np.float32)
    x[::block] = 127 * 2.0 ** -10
    xb = oracle.f32_to_bf16(x)
    xd = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
    S = plan.shard
    nbs = -(-S // block)
    codes = torch.zeros(plan.padded, dtype=torch.int8, device="cuda")
    scales = torch.zeros(n_d * nbs, device="cuda")
    gathered = torch.zeros(psi, dtype=torch.bfloat16, device="cuda")
    z.zero_quant_gather(plan.handle, xd, block, codes, scales, gathered)
    oc, osc, og = oracle.quant_gather(xb, n_d, psi, S, block)
    assert np.all(osc == np.float32(2.0 ** -10))
    assert np.array_equal(codes.cpu().numpy(), oc) and np.array_equal(u16(gathered), og)


@pytest.mark.parametrize("n_d,psi", [(3, 5), (4, 50_001), (2, 8192 * 3 + 1)])
def test_largest_shard_pad(n_d, psi):
    # shard_pad 4096: shards padded to a whole tile, trailing shards empty or short
    job = Job(psi, n_d, pad=4096, hp=z.hparams(lr=1e-3, weight_decay=0.1, max_norm=0.5), seed=17)
    for step in (1, 2):
        job.new_grads(step)
        job.gpu_step()
        job.oracle_step()
        job.settle()


def _with_subnormals(g, rng, frac=0.05):
    """Replace a fraction of a [n_d, row] bf16 tensor's entries by bf16
    subnormals (exponent field zero) of random sign and mantissa."""
    bits = g.view(torch.int16).numpy()
    mask = rng.random(bits.shape) < frac
    sub = (rng.integers(1, 128, size=bits.shape) | (rng.integers(0, 2, size=bits.shape) << 15)).astype(np.int16)
    bits[mask] = sub[mask]
    return g


@pytest.mark.parametrize("stage", [2, 3])
def test_subnormal_gradients(stage):
    # bf16 subnormals in every rank: the rank sums (mixed-precision adds)
    # and Adam must keep them as the oracle's IEEE arithmetic does
    n_d, psi = 4, 300_007
    job = Job(psi, n_d, stage=stage, pad=8, hp=z.hparams(lr=1e-3), seed=23)
    rng = np.random.default_rng(5)
    for step in (1, 2):
        g = synth.rank_grads(n_d, psi, 1e-36, 23, step, row_pad=job.buf.grads.shape[1] - psi)
        g = _with_subnormals(g, rng)
        job.buf.grads.copy_(g.cuda())
        job.rows = [u16(g[r, :psi]) for r in range(n_d)]
        assert any((np.asarray(r) & 0x7F80 == 0).any() and (np.asarray(r) & 0x7F).any() for r in job.rows)
        job.gpu_step()
        job.oracle_step()
        job.assert_bit_exact()


def test_subnormal_values_through_the_quantizers():
    # blocks whose values are bf16 subnormals (scale itself subnormal: the
    # exact path) next to blocks with a normal maximum and subnormal members
    n_d, psi = 2, 2048 * 8
    plan = z.Plan(psi, n_d, stage=2, shard_pad=8)
    S = plan.shard
    rng = np.random.default_rng(9)
    g = torch.zeros(n_d, z.row_len(psi), dtype=torch.bfloat16)
    g[:, :psi] = torch.from_numpy(rng.normal(0, 1e-37, size=(n_d, psi)).astype(np.float32)).to(torch.bfloat16)
    g = _with_subnormals(g, rng, frac=0.5)
    g[:, 2048 * 2:2048 * 3] = torch.from_numpy(rng.normal(0, 1e-3, size=(n_d, 2048)).astype(np.float32)).to(
        torch.bfloat16)
    g[:, 2048 * 2 + 7] = 3e-36   # a normal block maximum small enough that members may round to code 1
    gd = g.cuda()
    nbs = -(-S // 2048)
    n_dp = (n_d + 3) // 4 * 4
    codes = torch.zeros(n_d, (psi + 15) // 16 * 16, dtype=torch.int8, device="cuda")
    scales = torch.zeros(n_d * nbs * n_dp, device="cuda")
    z.zero_quantize_grads(plan.handle, [gd[r] for r in range(n_d)], 2048, [codes[r] for r in range(n_d)], scales)
    rows = [u16(g[r, :psi]) for r in range(n_d)]
    oc, osc = oracle.quantize_ranks(rows, psi, S, 2048)
    got_c = codes.cpu().numpy()
    for q in range(n_d):
        assert np.array_equal(got_c[q, :psi], oc[q][:psi])
    assert np.array_equal(u32(scales.cpu().numpy().reshape(osc.shape)), u32(osc))
    # the standalone quantized gather of the same values as one shard set
    x = gd[0, :psi].contiguous()
    qc = torch.zeros(psi, dtype=torch.int8, device="cuda")
    qs = torch.zeros(n_d * nbs, device="cuda")
    qg = torch.zeros(psi, dtype=torch.bfloat16, device="cuda")
    z.zero_quant_gather(plan.handle, x, 2048, qc, qs, qg)
    wc, ws, wg = oracle.quant_gather(u16(x), n_d, psi, S, 2048)
    assert np.array_equal(qc.cpu().numpy(), wc)
    assert np.array_equal(u32(qs.cpu().numpy()), u32(ws))
    assert np.array_equal(u16(qg), wg)
