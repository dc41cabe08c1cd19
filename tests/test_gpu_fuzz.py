"""Seeded random configurations of the fused step, each two steps on the GPU
and in the oracle: rank count, size, shard padding, stage, gradient and
parameter dtypes, clipping, weight decay, fp16 loss scaling (in place and
out of place), bucketing and gradient accumulation drawn together, so that
combinations no hand-written case covers are checked too."""
import numpy as np
import pytest

import oracle
import zero_optimizer_step_02_gb300 as z
from gpu_helpers import ORACLE_DT, Job, accum_ghat, oracle_hp

pytestmark = pytest.mark.gpu


def _draw(seed):
    rng = np.random.default_rng(1000 + seed)
    n_d = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 9, 16, 17, 32, 64]))
    psi = int(rng.choice([1, 7, 1000, 4095, 4096, 4097, 70_001, 300_007, 1_000_003]))
    pad = int(rng.choice([1, 8, 16, 64, 4096]))
    stage = int(rng.choice([1, 2, 3]))
    fp16 = bool(rng.random() < 0.35)
    ls = fp16 and bool(rng.random() < 0.6)
    return dict(n_d=n_d, psi=psi, pad=pad, stage=stage, fp16=fp16, ls=ls,
                pdt_fp16=bool(rng.random() < 0.25), clip=float(rng.choice([0.0, 0.0, 0.05, 1e3])),
                wd=float(rng.choice([0.0, 0.1])), pingpong=bool(rng.random() < 0.5),
                bucket=int(rng.choice([0, 0, 3 * 4096 + 5])), k=int(rng.choice([1, 1, 2, 3])))


@pytest.mark.parametrize("seed", range(24))
def test_random_configuration(seed):
    c = _draw(seed)
    gdt = z.ZERO_FP16 if c["fp16"] else z.ZERO_BF16
    pdt = z.ZERO_FP16 if c["pdt_fp16"] else None
    scale = 1024.0 if c["ls"] else 1.0
    hp = z.hparams(lr=1e-3, beta2=0.99, weight_decay=c["wd"], max_norm=c["clip"], loss_scaling=c["ls"],
                   scale_window=1000)
    job = Job(c["psi"], c["n_d"], stage=c["stage"], pad=c["pad"], gdt=gdt, pdt=pdt, hp=hp, seed=seed,
              pingpong=c["pingpong"], loss_scale=scale, bucket=c["bucket"])
    k = c["k"]
    for step in (1, 2):
        acc = None
        for mu in range(1, k + 1):
            job.new_grads(100 * step + mu, sigma=1e-2, scale=scale)
            if mu < k:
                job.buf.accumulate(first=mu == 1)
                acc = oracle.accumulate_grads(job.rows, ORACLE_DT[gdt], acc)
        b = job.buf
        if c["pingpong"]:
            z.zero_step_fused_accum(job.plan.handle, hp, b.rank_list(), None if k == 1 else b.acc, k, b.master, b.m, b.v,
                                    b.master2, b.m2, b.v2, b.lp, b.scalars, b.ws)
            b.master, b.master2 = b.master2, b.master
            b.m, b.m2 = b.m2, b.m
            b.v, b.v2 = b.v2, b.v
        else:
            z.zero_step_fused_accum(job.plan.handle, hp, b.rank_list(), None if k == 1 else b.acc, k, b.master, b.m,
                                    b.v, b.master, b.m, b.v, b.lp, b.scalars, b.ws)
        job.snapshot()
        skipped = oracle.zero_step_accum(job.rows, ORACLE_DT[gdt], acc, k, oracle_hp(hp), job.ost, c["pad"],
                                         c["stage"], param_dtype=ORACLE_DT[job.pdt], lp_shards=job.o_lp_shards,
                                         gathered=job.o_gathered)
        sc = job.scalars()
        assert sc.t == job.ost.scalars.t and sc.status == 0, c
        job.settle(ghat=lambda: accum_ghat(job, acc, k), skipped=skipped)
