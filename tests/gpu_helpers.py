"""Helpers of the GPU parity tests: seeded inputs made once on the CPU, the
same bytes given to the CUDA path (through the C ABI) and to the oracle."""
import os

import numpy as np
import torch

import oracle
import zero_optimizer_step_02_gb300 as z
from zero_optimizer_step_02_gb300 import synth

TORCH_DT = {z.ZERO_BF16: torch.bfloat16, z.ZERO_FP16: torch.float16}
ORACLE_DT = {z.ZERO_BF16: oracle.BF16, z.ZERO_FP16: oracle.FP16}


def u16(t):
    """A 16-bit torch tensor (any device) as numpy uint16 bit patterns."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def u32(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


# Clipped steps whose clip coefficient came out one fp32 ulp away from the
# oracle's (the squared norm is summed in another order on the GPU): per test,
# [steps that took that branch, clipped steps checked].  conftest reports it
# at the end of the session.
ULP_BRANCH = {}


def _note_clipped_step(one_ulp):
    key = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    n = ULP_BRANCH.setdefault(key, [0, 0])
    n[0] += int(one_ulp)
    n[1] += 1


def coef_ulps(a, b):
    """Distance of two fp32 clip coefficients in units in the last place."""
    return abs(int(np.float32(a).view(np.int32)) - int(np.float32(b).view(np.int32)))


def oracle_hp(hp):
    return oracle.hparams(lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2, eps=hp.eps, weight_decay=hp.weight_decay,
                          max_norm=hp.max_norm, loss_scaling=bool(hp.loss_scaling), scale_window=hp.scale_window,
                          min_scale=hp.min_scale)


class Job:
    """One simulated job on both sides: GPU buffers and the oracle's state."""

    def __init__(self, psi, n_d, stage=2, pad=8, gdt=z.ZERO_BF16, pdt=None, hp=None, seed=1, pingpong=False,
                 loss_scale=1.0, bucket=0, row_extra=0):
        self.hp = hp if hp is not None else z.hparams()
        self.plan = z.Plan(psi, n_d, stage=stage, grad_dtype=gdt, shard_pad=pad, param_dtype=pdt,
                           reduce_bucket_elems=bucket)
        self.psi, self.n_d, self.stage, self.pad, self.gdt = psi, n_d, stage, pad, gdt
        self.pdt = self.plan.param_dtype
        self.seed = seed
        self.buf = z.StepBuffers(self.plan, self.hp, device="cuda", pingpong=pingpong, row_extra=row_extra)
        master = synth.master_init(self.plan.padded, psi, seed)
        self.buf.master.copy_(master.cuda())
        self.buf.init_scalars(loss_scale)
        sc = oracle.new_scalars(loss_scale)
        self.ost = oracle.State(master.numpy().copy(), np.zeros(self.plan.padded, np.float32),
                                np.zeros(self.plan.padded, np.float32), sc)
        self.o_lp_shards = np.zeros(self.plan.padded, np.uint16)
        self.o_gathered = np.zeros(psi, np.uint16)

    def new_grads(self, step, sigma=1e-3, heavy_tail=False, scale=1.0, inf_at=None):
        g = synth.rank_grads(self.n_d, self.psi, sigma, self.seed, step, dtype=TORCH_DT[self.gdt],
                             heavy_tail=heavy_tail, scale=scale, row_pad=self.buf.grads.shape[1] - self.psi)
        if inf_at is not None:
            r, j = inf_at
            g[r, j] = float("inf")
        self.buf.grads.copy_(g.cuda())
        self.rows = [u16(g[r, :self.psi]) for r in range(self.n_d)]
        return g

    def gpu_step(self):
        self.buf.step(self.hp)

    def snapshot(self):
        """Keep the oracle's state before a step: the one-ulp clip check
        re-runs the step's update from it."""
        self.pre = self.ost.copy()

    def ghat(self):
        """The oracle's reduced gradient of the latest rank gradients (n_d*S,
        global index, padding +0): the rank-ordered fp32 sum divided by n_d
        times the loss scale the step was taken with."""
        d = float(self.n_d) * (self.pre.scalars.loss_scale if self.hp.loss_scaling else 1.0)
        return oracle.reduce_scatter(self.rows, ORACLE_DT[self.gdt], d, self.plan.shard)

    def oracle_step(self):
        self.snapshot()
        return oracle.zero_step(self.rows, ORACLE_DT[self.gdt], oracle_hp(self.hp), self.ost, self.pad,
                                self.stage, param_dtype=ORACLE_DT[self.pdt], lp_shards=self.o_lp_shards,
                                gathered=self.o_gathered)

    def gpu_state(self):
        torch.cuda.synchronize()
        b = self.buf
        lp = u16(b.lp)[: (self.plan.padded if self.stage == 3 else self.psi)]
        return b.master.cpu().numpy(), b.m.cpu().numpy(), b.v.cpu().numpy(), lp

    def oracle_lp(self):
        return self.o_lp_shards if self.stage == 3 else self.o_gathered

    def assert_bit_exact(self, lp=True):
        """master/m/v bit for bit, and the 16-bit parameters unless lp=False
        (a step whose epilogue writes another output)."""
        gm, gmm, gv, glp = self.gpu_state()
        for name, a, b in (("master", gm, self.ost.master), ("m", gmm, self.ost.m), ("v", gv, self.ost.v)):
            bad = np.flatnonzero(u32(a) != u32(b))
            assert bad.size == 0, "%s differs at %d places, first %s: gpu %r oracle %r" % (
                name, bad.size, bad[:5], a[bad[:5]], b[bad[:5]])
        if not lp:
            return
        olp = self.oracle_lp()
        bad = np.flatnonzero(glp != olp[: glp.size])
        assert bad.size == 0, "16-bit params differ at %d places, first %s" % (bad.size, bad[:5])

    def assert_within_tolerance(self, rel=1e-6, lp_ulp=1, lp=True):
        """The stated tolerance: per array max|gpu - cpu| / max|cpu| <= rel,
        16-bit parameters (unless lp=False) within lp_ulp units in the last place."""
        gm, gmm, gv, glp = self.gpu_state()
        for name, a, b in (("master", gm, self.ost.master), ("m", gmm, self.ost.m), ("v", gv, self.ost.v)):
            denom = max(float(np.max(np.abs(b))), 1e-30)
            err = float(np.max(np.abs(a.astype(np.float64) - b.astype(np.float64)))) / denom
            assert err <= rel, "%s relative error %.3g > %.1g" % (name, err, rel)
        if not lp:
            return
        olp = self.oracle_lp()[: glp.size]
        # 16-bit patterns of same-sign values are ordered like the values
        d = np.abs(glp.astype(np.int64) - olp.astype(np.int64))
        same_sign = (glp >> 15) == (olp >> 15)
        assert np.all(d[same_sign] <= lp_ulp) and np.all(
            (glp[~same_sign] & 0x7FFF) + (olp[~same_sign] & 0x7FFF) <= lp_ulp)

    def scalars(self):
        torch.cuda.synchronize()
        return self.buf.scalars_host()

    def settle(self, ghat=None, lp=True, skipped=False):
        """Check a step against the oracle step taken from the same state.

        Without clipping, or with clip coefficients that agree, every result
        is bit-exact.  With clipping the GPU sums the squared norm in another
        (compensated, tree) order than the oracle's sequential fp64 sum, so
        its coefficient may be one fp32 ulp away; then the GPU's results are
        the step with that coefficient, and the check is complete all the
        same: the oracle's own Adam is re-run from the state before the step
        on its reduced gradient times the GPU's coefficient (applied when
        below one, as the clipping rule says), and master, m, v and the
        16-bit parameters must equal the GPU's bit for bit.  The oracle's
        state then takes that run's values, so the next step is again
        compared bit for bit.  ghat: a callable giving the oracle's reduced
        gradient (n_d*S), default Job.ghat.  Returns True when the one-ulp
        branch was taken."""
        if not (self.hp.max_norm > 0.0) or skipped:
            self.assert_bit_exact(lp=lp)
            return False
        sc = self.scalars()
        o = np.float32(self.ost.scalars.clip_coef)
        d = coef_ulps(sc.clip_coef, o)
        assert d <= 1, "clip coefficients %r (gpu) and %r (oracle) differ by %d ulp" % (sc.clip_coef, o, d)
        _note_clipped_step(d == 1)
        if d == 0:
            self.assert_bit_exact(lp=lp)
            return False
        self.redo_with_coef(np.float32(sc.clip_coef), (ghat or self.ghat)())
        self.assert_bit_exact(lp=lp)
        return True

    def redo_with_coef(self, coef, g_hat):
        """The oracle's update from the state before the step, with the
        given clip coefficient (see settle); replaces the oracle's state and
        16-bit outputs by its results."""
        after = self.ost.scalars   # t and the beta powers of the committed step
        st, lp = step_with_coef(self.pre, g_hat, coef, oracle_hp(self.hp), after.beta1_pow, after.beta2_pow,
                                self.psi, ORACLE_DT[self.pdt])
        self.ost.master, self.ost.m, self.ost.v = st.master, st.m, st.v
        self.ost.scalars.clip_coef = float(coef)
        self.o_lp_shards[:self.psi] = lp
        self.o_gathered[:self.psi] = lp


def accum_ghat(job, acc, k):
    """The oracle's reduced gradient of an accumulated step: the carry of
    micro-batches 1..k-1 plus the k-th micro-batch's rank sum (the oracle's
    accumulation), divided once by n_d * k times the loss scale the step was
    taken with (one IEEE fp32 division, as the accumulation reading states)."""
    total = oracle.accumulate_grads(job.rows, ORACLE_DT[job.gdt], acc)
    scale = job.pre.scalars.loss_scale if job.hp.loss_scaling else 1.0
    return total / (np.float32(job.n_d * k) * np.float32(scale))


def step_with_coef(pre, g_hat, coef, ohp, beta1_pow_t, beta2_pow_t, psi, pdt):
    """The oracle's Adam update of one step with a given clip coefficient:
    g = g_hat * coef (one fp32 multiplication, only when coef < 1, as the
    clipping rule applies it), then the oracle's Adam on [0, psi) of a copy
    of the state `pre`, with the committed step's beta powers, then the
    oracle's 16-bit cast.  Returns (state, 16-bit parameters [psi])."""
    st = pre.copy()
    g = np.ascontiguousarray(g_hat[:psi], dtype=np.float32)
    coef = np.float32(coef)
    if coef < np.float32(1.0):
        g = g * coef
    c = oracle.adam_consts(ohp, beta1_pow_t, beta2_pow_t)
    oracle.adam_update(ohp, c, g, st.master[:psi], st.m[:psi], st.v[:psi])
    return st, oracle.f32_to_lp(st.master[:psi], pdt)
