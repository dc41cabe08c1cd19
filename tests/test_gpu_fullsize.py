"""Parity at the workloads' full sizes, in the launch configuration the bench
times (the same plans and entry points), on sampled outputs the oracle
computes element by element.  Global quantities come from the oracle over
the whole input (the clipping norm) or from properties fixed by the inputs
(exactly one injected non-finite value).

Workloads (seeded synthetic inputs from zero_optimizer_step_02_gb300.synth):
  GPT-2-small ZeRO-2, Psi = 124,439,808, N_d = 8, AdamW, clip 1.0, heavy tail
  GPT-2-1.5B ZeRO-2, Psi = 1.5e9, N_d = 8, fp16 grads, loss scale 1024, skip
  Llama-3-8B-shaped ZeRO-3 layer, Psi_l = 218,112,000, N_d = 16 (also the
  8-layer loop, and the layer's quantized weight gather)
  Psi = 2^28 sweep ends, N_d = 2 (with the fused int8 gather) and N_d = 64
"""
import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_02_gb300 as z
from gpu_helpers import _note_clipped_step, coef_ulps, oracle_hp, u16, u32
from zero_optimizer_step_02_gb300 import synth

pytestmark = pytest.mark.gpu

NSAMPLE = 20_000


def _free_gb():
    free, _ = torch.cuda.mem_get_info()
    return free / 1e9


def _sample(psi, seed):
    rng = np.random.default_rng(seed)
    idx = rng.choice(psi, size=NSAMPLE, replace=False)
    edge = np.array([0, 1, 2047, 2048, psi // 2, psi - 2049, psi - 2048, psi - 1])
    return np.unique(np.concatenate([idx, edge[(edge >= 0) & (edge < psi)]]))


class FullJob:
    def __init__(self, psi, n_d, stage, gdt, hp, seed, pingpong=False, loss_scale=1.0, param_dtype=None):
        self.plan = z.Plan(psi, n_d, stage=stage, grad_dtype=gdt, shard_pad=8, param_dtype=param_dtype)
        self.hp, self.psi, self.n_d, self.seed = hp, psi, n_d, seed
        self.gdt = gdt
        self.buf = z.StepBuffers(self.plan, hp, device="cuda", pingpong=pingpong)
        self.buf.master.copy_(synth.master_init(self.plan.padded, psi, seed, device="cuda"))
        self.buf.init_scalars(loss_scale)
        self.osc = oracle.new_scalars(loss_scale)

    def fill_grads(self, step, sigma, heavy_tail=False, scale=1.0):
        for r in range(self.n_d):
            synth.gaussian_(self.buf.grads[r, :self.psi], sigma, self.seed, step, r, heavy_tail=heavy_tail,
                            scale=scale)

    def take(self, idx):
        ii = torch.from_numpy(idx).cuda()
        rows = [u16(self.buf.grads[r][ii]) for r in range(self.n_d)]
        st = [t[ii].cpu().numpy().copy() for t in (self.buf.master, self.buf.m, self.buf.v)]
        return rows, st

    def oracle_sampled(self, rows, st, divisor, coef=None):
        """The oracle's update of the sampled elements: rank-ordered mean,
        optional clip coefficient, Adam with the step's bias corrections."""
        odt = oracle.FP16 if self.gdt == z.ZERO_FP16 else oracle.BF16
        g = oracle.all_reduce_mean(rows, odt, divisor)
        if coef is not None:
            g = (g * np.float32(coef)).astype(np.float32)
        hp = oracle_hp(self.hp)
        b1 = self.osc.beta1_pow * float(np.float32(hp.beta1))
        b2 = self.osc.beta2_pow * float(np.float32(hp.beta2))
        c = oracle.adam_consts(hp, b1, b2)
        p, m, v = (a.copy() for a in st)
        oracle.adam_update(hp, c, g, p, m, v)
        self.osc.beta1_pow, self.osc.beta2_pow, self.osc.t = b1, b2, self.osc.t + 1
        return p, m, v

    def check(self, idx, want, lp_dtype=oracle.BF16):
        ii = torch.from_numpy(idx).cuda()
        got = [t[ii].cpu().numpy() for t in (self.buf.master, self.buf.m, self.buf.v)]
        lp = u16(self.buf.lp[ii])
        for name, a, b in zip(("master", "m", "v"), got, want):
            bad = np.flatnonzero(u32(a) != u32(b))
            assert bad.size == 0, "%s: %d of %d sampled elements differ" % (name, bad.size, idx.size)
        assert np.array_equal(lp, oracle.f32_to_lp(want[0], lp_dtype))


def test_gpt2_small_clip_full_size():
    psi, n_d = 124_439_808, 8
    hp = z.hparams(lr=3e-4, beta1=0.9, beta2=0.95, weight_decay=0.1, max_norm=1.0)
    job = FullJob(psi, n_d, 2, z.ZERO_BF16, hp, seed=202)
    idx = _sample(psi, 1)
    for step in (1, 2):
        job.fill_grads(step, 1e-2, heavy_tail=True)
        rows, st = job.take(idx)
        # the clip coefficient needs the norm over all of psi: the oracle's
        # reduce and sequential fp64 sum over the full gradient
        full = [u16(job.buf.grads[r, :psi]) for r in range(n_d)]
        g_full = oracle.all_reduce_mean(full, oracle.BF16, float(n_d))
        sq = oracle.sqnorm(g_full)
        del full, g_full
        coef, applied = oracle.clip_coef(1.0, sq)
        assert applied
        job.buf.step(hp)
        sc = job.buf.scalars_host()
        # the oracle's sequential fp64 sum carries up to (n - 1) * 2^-53 relative error
        assert sc.sqnorm == pytest.approx(sq, rel=2 * psi * 2.0 ** -53)
        # the coefficients may be one ulp apart (the norm is summed in another
        # order); the sampled elements are then the oracle's update with the
        # GPU's coefficient, bit for bit
        d = coef_ulps(sc.clip_coef, coef)
        assert d <= 1
        _note_clipped_step(d == 1)
        want = job.oracle_sampled(rows, st, float(n_d), coef if d == 0 else np.float32(sc.clip_coef))
        job.check(idx, want)


def test_gpt2_xl_fp16_loss_scale_full_size():
    psi, n_d = 1_500_000_000, 8
    if _free_gb() < 70:
        pytest.skip("needs ~64 GB of free device memory")
    hp = z.hparams(lr=1e-4, loss_scaling=True)
    job = FullJob(psi, n_d, 2, z.ZERO_FP16, hp, seed=303, pingpong=True, loss_scale=1024.0)
    idx = _sample(psi, 2)
    job.fill_grads(1, 1e-4, scale=1024.0)
    rows, st = job.take(idx)
    job.buf.step(hp)
    sc = job.buf.scalars_host()
    assert sc.overflow == 0 and sc.t == 1
    want = job.oracle_sampled(rows, st, float(n_d) * 1024.0)
    job.check(idx, want)
    # step 2: one rank carries +inf at one index -> skipped, scale halves
    job.fill_grads(2, 1e-4, scale=1024.0)
    r, j = synth.pick_index(303, 2, n_d, psi)
    job.buf.grads[r, j] = float("inf")
    job.buf.step(hp)
    sc = job.buf.scalars_host()
    assert sc.overflow == 1 and sc.t == 1 and sc.loss_scale == 512.0 and sc.good_steps == 0
    job.check(idx, want)   # the state (now in the other buffer set) is unchanged


@pytest.mark.parametrize("stage", [1, 2])
def test_gpt2_xl_fp16_parameters_full_size(stage):
    # the pages pair fp16 parameters with fp16 gradients (DP-notes, "Memory
    # Consumption Analysis"): the same workload with fp16 16-bit parameters,
    # as ZeRO-1 and ZeRO-2 (the same math), in place (a check pass, then the
    # guarded update), two steps on sampled elements
    psi, n_d = 1_500_000_000, 8
    if _free_gb() < 70:
        pytest.skip("needs ~64 GB of free device memory")
    hp = z.hparams(lr=1e-4, loss_scaling=True)
    job = FullJob(psi, n_d, stage, z.ZERO_FP16, hp, seed=313 + stage, loss_scale=1024.0, param_dtype=z.ZERO_FP16)
    assert job.buf.lp.dtype == torch.float16
    idx = _sample(psi, 5)
    for step in (1, 2):
        job.fill_grads(step, 1e-4, scale=1024.0)
        rows, st = job.take(idx)
        job.buf.step(hp)
        sc = job.buf.scalars_host()
        assert sc.overflow == 0 and sc.t == step and sc.status == 0
        want = job.oracle_sampled(rows, st, float(n_d) * 1024.0)
        job.check(idx, want, lp_dtype=oracle.FP16)


def test_llama_layer_zero3_full_size():
    psi, n_d = 218_112_000, 16   # one Llama-3-8B-shaped decoder layer
    hp = z.hparams(lr=1e-3)
    job = FullJob(psi, n_d, 3, z.ZERO_BF16, hp, seed=404)
    idx = _sample(psi, 3)
    S = job.plan.shard
    gathered = torch.zeros(psi, dtype=torch.bfloat16, device="cuda")
    for step in (1, 2):
        # gather the layer's bf16 shards (as written by the previous step)
        z.zero_all_gather(job.plan.handle, [job.buf.lp[r * S:(r + 1) * S] for r in range(n_d)], gathered,
                          job.buf.scalars)
        ii = torch.from_numpy(idx).cuda()
        assert torch.equal(gathered[ii], job.buf.lp[ii])
        job.fill_grads(step, 1e-3)
        rows, st = job.take(idx)
        job.buf.step(hp)
        want = job.oracle_sampled(rows, st, float(n_d))
        job.check(idx, want)
    assert job.buf.scalars_host().status == 0


def test_llama_8_layers_zero3_layer_loop_full_size():
    # the default bench workload in its launch configuration: 8 Llama-3-8B-
    # shaped layers (Psi_l = 218,112,000), N_d = 16, one zero_step_layers call
    # per step with the gathers on a second stream and two gathered buffers;
    # every layer's sampled elements against the oracle, the gathered values
    # of the last two layers against the shards the step started from
    psi, n_d, L = 218_112_000, 16, 8
    if _free_gb() < 100:
        pytest.skip("needs ~90 GB of free device memory")
    hp = z.hparams(lr=1e-3)
    jobs = [FullJob(psi, n_d, 3, z.ZERO_BF16, hp, seed=440 + l) for l in range(L)]
    scalars = torch.zeros(256, dtype=torch.uint8, device="cuda")
    z.zero_scalars_init(scalars)
    stack = z.LayerStack([(j.plan.handle, j.buf.rank_ptrs(), j.buf.master, j.buf.m, j.buf.v, j.buf.lp) for j in jobs])
    gathered = [torch.zeros(psi, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    idx = _sample(psi, 9)
    ii = torch.from_numpy(idx).cuda()
    for step in (1, 2):
        taken, before = [], []
        for j in jobs:
            j.fill_grads(step, 1e-3)
            taken.append(j.take(idx))
            before.append(j.buf.lp[ii].clone())
        z.zero_step_layers(hp, stack, 1, gathered, scalars, gather_stream=torch.cuda.Stream())
        torch.cuda.synchronize()
        assert z.read_scalars(scalars).t == step
        for l, j in enumerate(jobs):
            rows, st = taken[l]
            j.check(idx, j.oracle_sampled(rows, st, float(n_d)))
        # layers 6 and 7 were the last gathered into buffers 0 and 1: the
        # shards as the step found them
        for l in (L - 2, L - 1):
            assert torch.equal(gathered[l % 2][ii].view(torch.int16), before[l].view(torch.int16))
    assert z.read_scalars(scalars).status == 0


@pytest.mark.parametrize("n_d", [2, 4, 8, 16, 64])
def test_psi_2_28_full_size(n_d):
    psi = 1 << 28
    if _free_gb() < 2 * n_d * psi / 1e9 + 20:
        pytest.skip("not enough free device memory")
    hp = z.hparams(lr=1e-3)
    job = FullJob(psi, n_d, 2, z.ZERO_BF16, hp, seed=505 + n_d)
    idx = _sample(psi, 4)
    job.fill_grads(1, 1e-3)
    rows, st = job.take(idx)
    job.buf.step(hp)
    want = job.oracle_sampled(rows, st, float(n_d))
    job.check(idx, want)


def test_psi_2_28_fused_quantized_gather_full_size():
    psi, n_d = 1 << 28, 2
    hp = z.hparams(lr=1e-3)
    job = FullJob(psi, n_d, 2, z.ZERO_BF16, hp, seed=606)
    S = job.plan.shard
    nbs = -(-S // 2048)
    codes = torch.zeros(job.plan.padded, dtype=torch.int8, device="cuda")
    scales = torch.zeros(n_d * nbs, device="cuda")
    gathered = torch.zeros(psi, dtype=torch.bfloat16, device="cuda")
    # sample whole quantization blocks (the scale needs the whole block)
    rng = np.random.default_rng(5)
    blocks = np.unique(np.concatenate([rng.choice(n_d * nbs, 40, replace=False), [0, n_d * nbs - 1]]))
    idx = np.concatenate([np.arange(b // nbs * S + (b % nbs) * 2048, b // nbs * S + (b % nbs) * 2048 + 2048)
                          for b in blocks])
    job.fill_grads(1, 1e-3)
    rows, st = job.take(idx)
    b = job.buf
    z.zero_step_fused_qgather(job.plan.handle, hp, b.rank_list(), b.master, b.m, b.v, b.master, b.m, b.v, 2048,
                              codes, scales, gathered, b.scalars, b.ws)
    want = job.oracle_sampled(rows, st, float(n_d))
    ii = torch.from_numpy(idx).cuda()
    assert np.array_equal(u32(b.master[ii].cpu().numpy()), u32(want[0]))
    lp = oracle.f32_to_bf16(want[0])
    got_codes = codes[ii].cpu().numpy()
    got_g = u16(gathered[ii])
    got_s = scales[torch.from_numpy(blocks).cuda()].cpu().numpy()
    for k in range(blocks.size):
        sl = slice(k * 2048, (k + 1) * 2048)
        c, s, d = oracle.quantize_block(lp[sl])
        assert got_s[k] == np.float32(s)
        assert np.array_equal(got_codes[sl], c) and np.array_equal(got_g[sl], d)


@pytest.mark.parametrize("n_d", [8, 64])
def test_psi_2_28_quantized_gradient_exchange_full_size(n_d):
    # the bench's qgZ workload: sender on every rank, then the fused receiver
    # step; sampled elements against the oracle's point-wise reconstruction
    psi = 1 << 28
    if _free_gb() < n_d * psi * 3 / 1e9 + 20:
        pytest.skip("not enough free device memory")
    hp = z.hparams(lr=1e-3)
    job = FullJob(psi, n_d, 2, z.ZERO_BF16, hp, seed=707 + n_d)
    job.plan = z.Plan(psi, n_d, stage=2, grad_dtype=z.ZERO_BF16, shard_pad=16)
    S = job.plan.shard
    nbs = -(-S // 2048)
    n_dp = (n_d + 3) // 4 * 4
    codes = torch.empty(n_d, (psi + 15) // 16 * 16, dtype=torch.int8, device="cuda")
    scales = torch.empty(n_d * nbs * n_dp, device="cuda")
    idx = _sample(psi, 6)
    job.fill_grads(1, 1e-3)
    b = job.buf
    z.zero_quantize_grads(job.plan.handle, b.rank_list(), 2048, [codes[r] for r in range(n_d)], scales)
    ii = torch.from_numpy(idx).cuda()
    st = [t[ii].cpu().numpy().copy() for t in (b.master, b.m, b.v)]
    z.zero_step_fused_qgz(job.plan.handle, hp, [codes[r] for r in range(n_d)], scales, 2048, b.master, b.m, b.v,
                          b.master, b.m, b.v, b.lp, b.scalars)
    # the sender's codes at the samples are the oracle's: quantize the sampled
    # blocks on the CPU from the same bf16 bytes
    rows = (idx // S) * nbs + (idx % S) // 2048
    sc_all = scales.view(-1, n_dp).cpu().numpy()
    c_at = [codes[q][ii].cpu().numpy() for q in range(n_d)]
    s_at = [sc_all[rows, q] for q in range(n_d)]
    for blk in np.unique(rows)[:24]:
        r, bb = divmod(int(blk), nbs)
        lo = r * S + bb * 2048
        hi = min(lo + 2048, psi, (r + 1) * S)
        for q in (0, n_d - 1):
            x = u16(b.grads[q, lo:hi])
            oc, osc, _ = oracle.quantize_block(x)
            assert osc == sc_all[blk, q]
            assert np.array_equal(codes[q, lo:hi].cpu().numpy(), oc)
    g = oracle.reduce_points_q(c_at, s_at, float(n_d))
    hpo = oracle_hp(hp)
    c = oracle.adam_consts(hpo, float(np.float32(hpo.beta1)), float(np.float32(hpo.beta2)))
    p, m, v = (a.copy() for a in st)
    oracle.adam_update(hpo, c, g, p, m, v)
    job.check(idx, (p, m, v))


def test_llama_layer_quantized_weight_gather_full_size():
    # the layer loop's qwZ gather at its full size (Psi_l = 218,112,000, N_d =
    # 16 shards of 13,632,000): the bulk-copy pipeline on every full aligned
    # block, the plain loads on each shard's last (partial) block; sampled
    # whole blocks against the oracle's block quantizer, every scale checked
    psi, n_d = 218_112_000, 16
    plan = z.Plan(psi, n_d, stage=3, shard_pad=8)
    S = plan.shard
    nbs = -(-S // 2048)
    shards = torch.zeros(plan.padded, dtype=torch.bfloat16, device="cuda")
    synth.gaussian_(shards[:psi], 0.02, 707, 0)
    shards[5 * S + 4096:5 * S + 6144] = 0.0          # an all-zero block: scale 0, codes 0
    codes = torch.full((plan.padded,), 77, dtype=torch.int8, device="cuda")
    scales = torch.full((n_d * nbs,), -1.0, device="cuda")
    gathered = torch.zeros(psi, dtype=torch.bfloat16, device="cuda")
    z.zero_quant_gather(plan.handle, shards, 2048, codes, scales, gathered)
    torch.cuda.synchronize()
    # every full block's scale: its absmax / 127 (one fp32 division), from the
    # bf16 values on the host
    full = (S // 2048) * 2048
    x = u16(shards).reshape(n_d, S)[:, :full].astype(np.uint32) << 16
    amax = np.abs(x.view(np.float32)).reshape(n_d, S // 2048, 2048).max(axis=2)
    want_s = (amax / np.float32(127.0)).astype(np.float32)
    got_s = scales.view(n_d, nbs)[:, :S // 2048].cpu().numpy()
    assert np.array_equal(u32(got_s), u32(want_s))
    # sampled whole blocks (full ones, each shard's last, the zero one) bit for bit
    rng = np.random.default_rng(17)
    picks = [(r, int(b)) for r in range(n_d) for b in rng.choice(S // 2048, 3, replace=False)]
    picks += [(r, nbs - 1) for r in range(n_d)] + [(5, 2)]
    for r, b in picks:
        lo = r * S + b * 2048
        hi = min(lo + 2048, r * S + S, psi)
        x = u16(shards[lo:hi])
        c, s, d = oracle.quantize_block(x)
        assert u32(np.float32(scales[r * nbs + b].item())) == u32(np.float32(s))
        assert np.array_equal(codes[lo:hi].cpu().numpy(), c)
        assert np.array_equal(u16(gathered[lo:hi]), d)
