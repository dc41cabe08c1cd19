"""GPU parity of the ZeRO++ variants under the step's global checks: the
int8 gather with global-norm clipping and with fp16 loss scaling (overflow
skip), and the quantized gradient exchange with clipping, against the oracle
(the plain step followed by the block quantizer; the quantized-exchange step)
on the same bytes."""
import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_02_gb300 as z
from gpu_helpers import Job, oracle_hp, u16, u32
from zero_optimizer_step_02_gb300 import synth

pytestmark = pytest.mark.gpu


class QGather:
    """The int8-gather outputs of a job and the oracle's quantizer over the
    oracle's updated 16-bit parameters."""

    def __init__(self, job):
        self.job = job
        S = job.plan.shard
        self.nbs = -(-S // 2048)
        self.codes = torch.zeros(job.plan.padded, dtype=torch.int8, device="cuda")
        self.scales = torch.full((job.n_d * self.nbs,), -1.0, device="cuda")
        self.gathered = torch.zeros(job.psi, dtype=torch.bfloat16, device="cuda")

    def gpu_step(self):
        j, b = self.job, self.job.buf
        z.zero_step_fused_qgather(j.plan.handle, j.hp, b.rank_ptrs(), b.master, b.m, b.v, b.master, b.m, b.v, 2048,
                                  self.codes, self.scales, self.gathered, b.scalars, b.ws)

    def assert_outputs(self):
        j = self.job
        lp_flat = np.zeros(j.plan.padded, np.uint16)
        lp_flat[:j.psi] = j.o_gathered
        oc, osc, og = oracle.quant_gather(lp_flat, j.n_d, j.psi, j.plan.shard, 2048)
        assert np.array_equal(self.codes.cpu().numpy()[:j.psi], oc[:j.psi])
        assert np.array_equal(u32(self.scales.cpu().numpy()), u32(osc))
        assert np.array_equal(u16(self.gathered), og)


@pytest.mark.parametrize("n_d,psi,pad", [(2, 300_001, 8), (8, 400_003, 8), (5, 123_457, 1), (8, 7, 8)])
def test_quantized_gather_with_clipping(n_d, psi, pad):
    hp = z.hparams(lr=3e-4, beta2=0.95, weight_decay=0.1, max_norm=1.0)
    job = Job(psi, n_d, pad=pad, hp=hp, seed=81 + n_d)
    q = QGather(job)
    for step in range(1, 4):
        job.new_grads(step, sigma=1e-2, heavy_tail=True)
        q.gpu_step()
        job.oracle_step()
        if psi >= 1000:
            assert np.float32(job.ost.scalars.clip_coef) < 1.0      # the clip is active
        # state bit for bit (with the GPU's coefficient if it is one ulp off),
        # then codes, scales and dequantized values bit for bit against the
        # oracle's quantizer over those updated 16-bit weights
        job.settle(lp=False)
        q.assert_outputs()
        assert job.scalars().t == step


@pytest.mark.parametrize("max_norm", [0.0, 1e-3])
def test_quantized_gather_overflow_skip(max_norm):
    # fp16 gradients with a loss scale, one +inf at step 3: that step writes
    # nothing (state, codes, scales and gathered values stay the previous
    # step's) and halves the scale
    psi, n_d = 250_003, 4
    hp = z.hparams(lr=1e-4, loss_scaling=True, max_norm=max_norm)
    job = Job(psi, n_d, gdt=z.ZERO_FP16, hp=hp, seed=83, loss_scale=1024.0)
    q = QGather(job)
    for step in range(1, 6):
        inf_at = synth.pick_index(83, step, n_d, psi) if step == 3 else None
        job.new_grads(step, sigma=1e-4, scale=job.ost.scalars.loss_scale, inf_at=inf_at)
        q.gpu_step()
        skipped = job.oracle_step()
        sc = job.scalars()
        assert bool(sc.overflow) == skipped == (step == 3)
        assert sc.loss_scale == job.ost.scalars.loss_scale and sc.t == job.ost.scalars.t
        job.settle(lp=False, skipped=skipped)
        q.assert_outputs()


# 13 and 14 ranks: either side of the largest rank count whose reduce pass
# over the codes runs two CTAs per SM (both rings in 228 KB of shared
# memory), with more tiles than two CTAs on every SM take at once
@pytest.mark.parametrize("n_d,psi,pad", [(2, 300_001, 16), (8, 400_003, 16), (17, 70_001, 1), (4, 5_000, 16),
                                         (8, 7, 16), (3, 1, 1), (13, 2_500_001, 16), (14, 2_500_001, 16)])
@pytest.mark.parametrize("stage", [2, 3])
def test_quantized_exchange_with_clipping(n_d, psi, pad, stage):
    # n_d <= 4: reduce pass over the codes, then the fused step re-reads them;
    # n_d > 4: the reduce pass writes the reduced gradient, the Adam pass reads it
    hp = z.hparams(lr=3e-4, beta2=0.95, weight_decay=0.1, max_norm=1.0)
    job = Job(psi, n_d, stage=stage, pad=pad, hp=hp, seed=91 + n_d)
    S = job.plan.shard
    row = (psi + 15) // 16 * 16
    codes = torch.full((n_d, row), 77, dtype=torch.int8, device="cuda")
    n_dp = (n_d + 3) // 4 * 4
    scales = torch.full((n_d * -(-S // 2048) * n_dp,), -1.0, device="cuda")
    b = job.buf
    for step in range(1, 4):
        job.new_grads(step, sigma=1e-2, heavy_tail=True)
        z.zero_quantize_grads(job.plan.handle, b.rank_ptrs(), 2048, [codes[r] for r in range(n_d)], scales)
        z.zero_step_fused_qgz(job.plan.handle, hp, [codes[r] for r in range(n_d)], scales, 2048, b.master, b.m, b.v,
                              b.master, b.m, b.v, b.lp, b.scalars, b.ws)
        oc, osc = oracle.quantize_ranks(job.rows, psi, S, 2048)
        job.snapshot()
        oracle.zero_step_qgz(oc, osc, 2048, oracle_hp(hp), job.ost, pad, stage, psi, lp_shards=job.o_lp_shards,
                             gathered=job.o_gathered)
        if psi >= 1000:
            assert np.float32(job.ost.scalars.clip_coef) < 1.0
        sc = job.scalars()
        assert sc.sqnorm == pytest.approx(job.ost.scalars.sqnorm, rel=2 * psi * 2.0 ** -53)
        job.settle(ghat=lambda: oracle.reduce_scatter_q(oc, osc, psi, S, 2048, float(n_d)))
        assert sc.t == step and sc.status == 0


def test_quantized_exchange_clipped_on_grid_equals_the_plain_clipped_step():
    # gradients on the int8 grid: the exchange is lossless, so the clipped
    # step from the codes gives the plain clipped step's bits
    n_d, psi, pad = 8, 4096 * 40, 16
    hp = z.hparams(lr=1e-3, max_norm=0.5)
    plan = z.Plan(psi, n_d, stage=2, shard_pad=pad)
    S = plan.shard
    rng = np.random.default_rng(5)
    k = rng.integers(-127, 128, size=(n_d, psi)).astype(np.float32)
    k[:, ::2048] = 127.0
    x = torch.from_numpy(k * 2.0 ** -10).to(torch.bfloat16)
    grads = torch.zeros(n_d, z.row_len(psi), dtype=torch.bfloat16)
    grads[:, :psi] = x
    a = z.StepBuffers(plan, hp, device="cuda", grads=grads.cuda())
    c = z.StepBuffers(plan, hp, device="cuda")
    master = synth.master_init(plan.padded, psi, seed=2, device="cuda")
    for s in (a, c):
        s.master.copy_(master)
        s.init_scalars()
    codes = torch.zeros(n_d, psi, dtype=torch.int8, device="cuda")
    scales = torch.zeros(n_d * -(-S // 2048) * ((n_d + 3) // 4 * 4), device="cuda")
    z.zero_quantize_grads(plan.handle, a.rank_ptrs(), 2048, [codes[r] for r in range(n_d)], scales)
    a.step(hp)
    z.zero_step_fused_qgz(plan.handle, hp, [codes[r] for r in range(n_d)], scales, 2048, c.master, c.m, c.v,
                          c.master, c.m, c.v, c.lp, c.scalars, c.ws)
    torch.cuda.synchronize()
    sa, scc = a.scalars_host(), c.scalars_host()
    assert sa.clip_coef < 1.0 and sa.clip_coef == scc.clip_coef
    assert torch.equal(a.master.view(torch.int32), c.master.view(torch.int32))
    assert torch.equal(a.lp.view(torch.int16), c.lp.view(torch.int16))
