"""Seeded random configurations of the ZeRO++ steps, two steps each on the
GPU and in the oracle: the int8 gather, the quantized gradient exchange, or
both, with the rank count, size, shard padding, stage, clipping and weight
decay drawn together."""
import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_02_gb300 as z
from gpu_helpers import Job, oracle_hp, u16, u32

pytestmark = pytest.mark.gpu


def _draw(seed):
    rng = np.random.default_rng(2000 + seed)
    mode = str(rng.choice(["qgather", "qgz", "both"]))
    return dict(mode=mode, n_d=int(rng.choice([1, 2, 3, 5, 8, 9, 16, 17, 32])),
                psi=int(rng.choice([1, 9, 2047, 2049, 4096, 40_001, 123_457, 300_007])),
                pad=int(rng.choice([1, 16, 64, 4096])), stage=int(rng.choice([2, 3])) if mode == "qgz" else 2,
                clip=float(rng.choice([0.0, 0.0, 0.05, 1e3])), wd=float(rng.choice([0.0, 0.1])))


@pytest.mark.parametrize("seed", range(16))
def test_random_zeropp_configuration(seed):
    c = _draw(seed)
    n_d, psi, pad = c["n_d"], c["psi"], c["pad"]
    hp = z.hparams(lr=1e-3, beta2=0.99, weight_decay=c["wd"], max_norm=c["clip"])
    job = Job(psi, n_d, stage=c["stage"], pad=pad, hp=hp, seed=300 + seed)
    S = job.plan.shard
    nbs = -(-S // 2048)
    b = job.buf
    codes = torch.full((n_d, (psi + 15) // 16 * 16), 77, dtype=torch.int8, device="cuda")
    scales = torch.full((n_d * nbs * ((n_d + 3) // 4 * 4),), -1.0, device="cuda")
    g_codes = torch.zeros(job.plan.padded, dtype=torch.int8, device="cuda")
    g_scales = torch.full((n_d * nbs,), -1.0, device="cuda")
    gathered = torch.zeros(psi, dtype=torch.bfloat16, device="cuda")
    rows = [codes[r] for r in range(n_d)]
    quant_out = c["mode"] != "qgz"
    for step in (1, 2):
        job.new_grads(step, sigma=1e-2, heavy_tail=True)
        ghat = None
        if c["mode"] == "qgather":
            z.zero_step_fused_qgather(job.plan.handle, hp, b.rank_ptrs(), b.master, b.m, b.v, b.master, b.m, b.v,
                                      2048, g_codes, g_scales, gathered, b.scalars, b.ws)
            job.oracle_step()
            lp_flat = np.zeros(job.plan.padded, np.uint16)
            lp_flat[:psi] = job.o_gathered
        else:
            z.zero_quantize_grads(job.plan.handle, b.rank_ptrs(), 2048, rows, scales)
            oc, osc = oracle.quantize_ranks(job.rows, psi, S, 2048)
            job.snapshot()
            ghat = lambda: oracle.reduce_scatter_q(oc, osc, psi, S, 2048, float(n_d))  # noqa: E731
            if c["mode"] == "qgz":
                z.zero_step_fused_qgz(job.plan.handle, hp, rows, scales, 2048, b.master, b.m, b.v, b.master, b.m,
                                      b.v, b.lp, b.scalars, b.ws)
                oracle.zero_step_qgz(oc, osc, 2048, oracle_hp(hp), job.ost, pad, c["stage"], psi,
                                     lp_shards=job.o_lp_shards, gathered=job.o_gathered)
            else:
                z.zero_step_fused_qgz_qgather(job.plan.handle, hp, rows, scales, 2048, b.master, b.m, b.v, b.master,
                                              b.m, b.v, g_codes, g_scales, gathered, b.scalars, b.ws)
                oracle.zero_step_qgz(oc, osc, 2048, oracle_hp(hp), job.ost, pad, 3, psi,
                                     lp_shards=job.o_lp_shards)
                lp_flat = job.o_lp_shards
        sc = job.scalars()
        assert sc.t == job.ost.scalars.t == step and sc.status == 0, c
        job.settle(ghat=ghat, lp=not quant_out)
        if quant_out:
            if c["mode"] == "qgather":
                lp_flat[:psi] = job.o_gathered      # the updated weights the step quantized
            qc, qs, qg = oracle.quant_gather(lp_flat, n_d, psi, S, 2048)
            assert np.array_equal(g_codes.cpu().numpy()[:psi], qc[:psi]), c
            assert np.array_equal(u32(g_scales.cpu().numpy()), u32(qs)), c
            assert np.array_equal(u16(gathered), qg), c
