"""GPU parity of the ZeRO++ step with both quantized exchanges in one pass:
the ranks' int8 gradient codes in (qgZ), the int8 gather of the updated
weights out (qwZ), against the oracle's quantized-exchange step followed by
its block quantizer, on the same bytes."""
import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_02_gb300 as z
from gpu_helpers import Job, oracle_hp, u16, u32

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n_d,psi,pad,clip", [(2, 300_001, 16, False), (8, 400_003, 16, True),
                                              (16, 200_003, 16, False), (17, 70_001, 1, True),
                                              (8, 100_000, 16, False), (32, 4097 * 7, 16, True),
                                              (8, 7, 16, True), (4, 2, 1, False)])
def test_two_exchange_step(n_d, psi, pad, clip):
    hp = z.hparams(lr=3e-4, beta2=0.95, weight_decay=0.1, max_norm=1.0 if clip else 0.0)
    job = Job(psi, n_d, pad=pad, hp=hp, seed=101 + n_d)
    S = job.plan.shard
    nbs = -(-S // 2048)
    n_dp = (n_d + 3) // 4 * 4
    codes = torch.full((n_d, (psi + 15) // 16 * 16), 77, dtype=torch.int8, device="cuda")
    scales = torch.full((n_d * nbs * n_dp,), -1.0, device="cuda")
    g_codes = torch.zeros(job.plan.padded, dtype=torch.int8, device="cuda")
    g_scales = torch.full((n_d * nbs,), -1.0, device="cuda")
    gathered = torch.zeros(psi, dtype=torch.bfloat16, device="cuda")
    b = job.buf
    code_rows = [codes[r] for r in range(n_d)]
    for step in range(1, 4):
        job.new_grads(step, sigma=1e-2, heavy_tail=True)
        z.zero_quantize_grads(job.plan.handle, b.rank_ptrs(), 2048, code_rows, scales)
        z.zero_step_fused_qgz_qgather(job.plan.handle, hp, code_rows, scales, 2048, b.master, b.m, b.v, b.master,
                                      b.m, b.v, g_codes, g_scales, gathered, b.scalars, b.ws)
        oc, osc = oracle.quantize_ranks(job.rows, psi, S, 2048)
        job.snapshot()
        oracle.zero_step_qgz(oc, osc, 2048, oracle_hp(hp), job.ost, pad, 3, psi, lp_shards=job.o_lp_shards)
        sc = job.scalars()
        assert sc.t == step and sc.status == 0
        # the state bit for bit (with the GPU's clip coefficient when it is one
        # ulp off the oracle's), then the int8 gather of those 16-bit weights
        job.settle(ghat=lambda: oracle.reduce_scatter_q(oc, osc, psi, S, 2048, float(n_d)), lp=False)
        qc, qs, qg = oracle.quant_gather(job.o_lp_shards, n_d, psi, S, 2048)
        assert np.array_equal(g_codes.cpu().numpy()[:psi], qc[:psi])
        assert np.array_equal(u32(g_scales.cpu().numpy()), u32(qs))
        assert np.array_equal(u16(gathered), qg)
