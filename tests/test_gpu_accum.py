"""GPU parity of gradient accumulation: k micro-batches per optimizer step,
each reduce-scattered into the fp32 accumulator (zero_accumulate_grads), the
step at the last one (zero_step_fused_accum) -- bit for bit against the
oracle on the same bytes, in every pass schedule of the step (plain, clipped
with the reduced gradient in HBM or re-read, loss scaling in place and
speculative, bucketed), plus the full-size GPT-2-small workload on samples."""
import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_02_gb300 as z
from gpu_helpers import ORACLE_DT, Job, accum_ghat, oracle_hp, u16, u32
from zero_optimizer_step_02_gb300 import synth

pytestmark = pytest.mark.gpu


class AccumJob(Job):
    """A Job whose steps take k micro-batches."""

    def micro_rows(self, step, mu, sigma=1e-3, heavy_tail=False, scale=1.0, inf_at=None):
        g = self.new_grads(1000 * step + mu, sigma=sigma, heavy_tail=heavy_tail, scale=scale, inf_at=inf_at)
        return g

    def run_step(self, step, k, **kw):
        """Both sides: k - 1 accumulations, then the step at micro-batch k."""
        acc = None
        for mu in range(1, k):
            self.micro_rows(step, mu, **kw)
            self.buf.accumulate(first=mu == 1)
            acc = oracle.accumulate_grads(self.rows, ORACLE_DT[self.gdt], acc)
        self.micro_rows(step, k, **kw)
        self.acc_k = (acc, k)
        if self.buf.pingpong:
            a = None if k == 1 else self.buf.acc
            b = self.buf
            z.zero_step_fused_accum(self.plan.handle, self.hp, b.rank_list(), a, k, b.master, b.m, b.v, b.master2,
                                    b.m2, b.v2, b.lp, b.scalars, b.ws)
            b.master, b.master2 = b.master2, b.master
            b.m, b.m2 = b.m2, b.m
            b.v, b.v2 = b.v2, b.v
        else:
            self.buf.step_accum(self.hp, k)
        self.snapshot()
        return oracle.zero_step_accum(self.rows, ORACLE_DT[self.gdt], acc, k, oracle_hp(self.hp), self.ost,
                                      self.pad, self.stage, param_dtype=ORACLE_DT[self.pdt],
                                      lp_shards=self.o_lp_shards, gathered=self.o_gathered), acc

    def assert_step(self, skipped=False):
        """Bit-exact; with clipping, against the oracle's update with the GPU's
        coefficient when the two coefficients are one ulp apart (Job.settle)."""
        acc, k = self.acc_k
        self.settle(ghat=lambda: accum_ghat(self, acc, k), skipped=skipped)


CASES = [  # (n_d, k, psi, pad, stage)
    (1, 2, 5000, 8, 2), (2, 4, 2047, 1, 2), (3, 3, 40_000, 8, 3), (4, 2, 1_000_003, 8, 2),
    (8, 4, 123_457, 8, 2), (16, 2, 70_001, 64, 3), (64, 2, 20_000, 8, 2), (5, 8, 3, 64, 1),
]


@pytest.mark.parametrize("n_d,k,psi,pad,stage", CASES)
def test_accumulator_bit_exact(n_d, k, psi, pad, stage):
    job = AccumJob(psi, n_d, stage=stage, pad=pad, seed=psi + k)
    acc = None
    for mu in range(1, k + 1):
        job.micro_rows(1, mu, sigma=1e-2, heavy_tail=True)
        job.buf.accumulate(first=mu == 1)
        acc = oracle.accumulate_grads(job.rows, oracle.BF16, acc)
    torch.cuda.synchronize()
    got = job.buf.acc[:psi].cpu().numpy()
    bad = np.flatnonzero(u32(got) != u32(acc))
    assert bad.size == 0, "accumulator differs at %d places, first %s" % (bad.size, bad[:5])
    # the padding past psi is not touched (it stays as allocated: zero)
    assert torch.count_nonzero(job.buf.acc[psi:]).item() == 0


def test_accumulate_separate_in_and_out():
    n_d, psi = 4, 300_007
    job = AccumJob(psi, n_d, seed=2)
    job.micro_rows(1, 1)
    job.buf.accumulate(first=True)
    first = job.buf.acc.clone()
    out = torch.full_like(first, -7.0)
    job.micro_rows(1, 2)
    z.zero_accumulate_grads(job.plan.handle, job.buf.rank_list(), first, out, job.buf.scalars)
    torch.cuda.synchronize()
    want = oracle.accumulate_grads(job.rows, oracle.BF16, first[:psi].cpu().numpy())
    assert np.array_equal(u32(out[:psi].cpu().numpy()), u32(want))
    assert torch.all(out[psi:] == -7.0)
    # the input is read only
    assert torch.equal(first, job.buf.acc)


@pytest.mark.parametrize("n_d,k,psi,pad,stage", CASES)
@pytest.mark.parametrize("variant", ["adamw", "clip"])
def test_accumulated_step(n_d, k, psi, pad, stage, variant):
    hp = z.hparams(lr=3e-4, beta2=0.95, weight_decay=0.1, max_norm=0.05 if variant == "clip" else 0.0)
    job = AccumJob(psi, n_d, stage=stage, pad=pad, hp=hp, seed=psi + n_d)
    for step in range(1, 4):
        skipped, _ = job.run_step(step, k, sigma=1e-2, heavy_tail=True)
        assert not skipped
        job.assert_step()
    assert job.scalars().t == 3


def test_one_micro_batch_equals_the_plain_step():
    hp = z.hparams(lr=1e-3, max_norm=0.1)
    a = Job(400_001, 8, hp=hp, seed=4)
    b = Job(400_001, 8, hp=hp, seed=4)
    for step in range(1, 3):
        a.new_grads(step)
        b.new_grads(step)
        a.gpu_step()
        b.buf.step_accum(hp, 1)
    torch.cuda.synchronize()
    for x, y in ((a.buf.master, b.buf.master), (a.buf.m, b.buf.m), (a.buf.v, b.buf.v), (a.buf.lp, b.buf.lp)):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))


@pytest.mark.parametrize("pingpong", [False, True])   # in place: check pass; out of place: speculative
def test_loss_scaling_with_an_overflow_in_an_early_micro_batch(pingpong):
    hp = z.hparams(lr=1e-4, loss_scaling=True, scale_window=2, min_scale=1.0)
    n_d, k, psi = 4, 3, 200_003
    job = AccumJob(psi, n_d, gdt=z.ZERO_FP16, hp=hp, seed=8, pingpong=pingpong, loss_scale=1024.0)
    for step in range(1, 6):
        inf_at = (2, 4097 * step) if step == 3 else None
        acc = None
        for mu in range(1, k):
            job.micro_rows(step, mu, sigma=1e-3, scale=job.ost.scalars.loss_scale,
                           inf_at=inf_at if mu == 1 else None)
            job.buf.accumulate(first=mu == 1)
            acc = oracle.accumulate_grads(job.rows, oracle.FP16, acc)
        job.micro_rows(step, k, sigma=1e-3, scale=job.ost.scalars.loss_scale)
        if pingpong:
            b = job.buf
            z.zero_step_fused_accum(job.plan.handle, hp, b.rank_list(), b.acc, k, b.master, b.m, b.v, b.master2,
                                    b.m2, b.v2, b.lp, b.scalars, b.ws)
            b.master, b.master2 = b.master2, b.master
            b.m, b.m2 = b.m2, b.m
            b.v, b.v2 = b.v2, b.v
        else:
            job.buf.step_accum(hp, k)
        skipped = oracle.zero_step_accum(job.rows, oracle.FP16, acc, k, oracle_hp(hp), job.ost, job.pad, job.stage,
                                         gathered=job.o_gathered)
        assert skipped == (step == 3)
        sc = job.scalars()
        assert sc.overflow == int(skipped) and sc.loss_scale == job.ost.scalars.loss_scale
        assert sc.t == job.ost.scalars.t
        job.assert_bit_exact()    # a skipped speculative step restored its out buffers from in


def test_bucketed_accumulated_step():
    # no global check: the step runs in buckets of the plan's bucket size
    hp = z.hparams(lr=1e-3, weight_decay=0.01)
    job = AccumJob(1_000_003, 8, hp=hp, seed=6, bucket=3 * 4096 + 5)
    for step in range(1, 3):
        job.run_step(step, 3)
        job.assert_bit_exact()


def test_fp16_parameters_and_gradients():
    hp = z.hparams(lr=1e-4)
    job = AccumJob(300_007, 4, gdt=z.ZERO_FP16, pdt=z.ZERO_FP16, hp=hp, seed=9)
    for step in range(1, 3):
        job.run_step(step, 4, sigma=1e-2)
        job.assert_bit_exact()


def test_argument_checks_need_no_launch():
    job = AccumJob(10_000, 2, seed=1)
    b = job.buf
    with pytest.raises(z.ZeroError):   # acc given with one micro-batch
        z.zero_step_fused_accum(job.plan.handle, job.hp, b.rank_list(), b.master, 1, b.master, b.m, b.v, b.master,
                                b.m, b.v, b.lp, b.scalars, b.ws)
    with pytest.raises(z.ZeroError):   # no acc with two
        z.zero_step_fused_accum(job.plan.handle, job.hp, b.rank_list(), None, 2, b.master, b.m, b.v, b.master,
                                b.m, b.v, b.lp, b.scalars, b.ws)
    acc = torch.zeros(job.plan.padded + 8, device="cuda")
    with pytest.raises(z.ZeroError):   # partly overlapping in and out
        z.zero_accumulate_grads(job.plan.handle, b.rank_list(), acc[:job.plan.padded], acc[4:4 + job.plan.padded])


# ------------------------------------------------------------- full size
NSAMPLE = 20_000


def test_gpt2_small_full_size_sampled():
    # GPT-2-small ZeRO-2, Psi = 124,439,808, N_d = 8, AdamW, k = 4 micro-batches,
    # in the bench's launch configuration; the oracle updates sampled elements
    psi, n_d, k = 124_439_808, 8, 4
    if torch.cuda.mem_get_info()[0] < 12e9:
        pytest.skip("needs 12 GB free")
    hp = z.hparams(lr=3e-4, beta1=0.9, beta2=0.95, weight_decay=0.1)
    plan = z.Plan(psi, n_d, stage=2, shard_pad=8)
    buf = z.StepBuffers(plan, hp, device="cuda")
    buf.master.copy_(synth.master_init(plan.padded, psi, 21, device="cuda"))
    buf.init_scalars()
    rng = np.random.default_rng(0)
    idx = np.unique(np.concatenate([rng.choice(psi, NSAMPLE, replace=False),
                                    [0, 1, 4095, 4096, psi // 2, psi - 4097, psi - 4096, psi - 1]]))
    ii = torch.from_numpy(idx).cuda()
    st = [t[ii].cpu().numpy().copy() for t in (buf.master, buf.m, buf.v)]
    acc = None
    for mu in range(1, k + 1):
        for r in range(n_d):
            synth.gaussian_(buf.grads[r, :psi], 1e-3, 21, mu, r, heavy_tail=True)
        rows = [u16(buf.grads[r][ii]) for r in range(n_d)]
        if mu < k:
            buf.accumulate(first=mu == 1)
            acc = oracle.accumulate_grads(rows, oracle.BF16, acc)
    buf.step_accum(hp, k)
    # the oracle's accumulated step on the sampled elements as a problem of
    # their own (every quantity is per element: no clipping here)
    n = idx.size
    S = oracle.shard_size(n, n_d, 1)
    ost = oracle.State(*[np.zeros(n_d * S, np.float32) for _ in range(3)], oracle.new_scalars())
    for dst, src in zip((ost.master, ost.m, ost.v), st):
        dst[:n] = src
    gathered = np.zeros(n, np.uint16)
    assert not oracle.zero_step_accum(rows, oracle.BF16, acc, k, oracle_hp(hp), ost, 1, 2, gathered=gathered)
    torch.cuda.synchronize()
    got = [t[ii].cpu().numpy() for t in (buf.master, buf.m, buf.v)]
    for name, a, b in zip(("master", "m", "v"), got, (ost.master, ost.m, ost.v)):
        bad = np.flatnonzero(u32(a) != u32(b[:n]))
        assert bad.size == 0, "%s differs at %d sampled places" % (name, bad.size)
    assert np.array_equal(u16(buf.lp[ii]), gathered)
    assert buf.scalars_host().t == 1
