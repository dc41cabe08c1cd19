"""Robustness of the CUDA path: checkpoint and resume are exact, no kernel
writes outside its buffers (canary guard zones), and the ZeRO-3 layer-wise
loop (gather each layer's shards, then the step) matches the oracle."""
import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_02_gb300 as z
from gpu_helpers import Job, oracle_hp, u16, u32
from zero_optimizer_step_02_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("hp_kw", [dict(lr=1e-3), dict(lr=3e-4, beta2=0.95, weight_decay=0.1, max_norm=1.0)])
def test_checkpoint_resume_is_bitwise(hp_kw):
    # the step's state is {master, m, v} plus the 64-byte scalars block (t,
    # beta powers, loss scale, counters): saving and restoring those resumes
    # the run exactly
    psi, n_d = 300_007, 8
    hp = z.hparams(**hp_kw)
    run = Job(psi, n_d, hp=hp, seed=7)
    for step in range(1, 7):
        run.new_grads(step, sigma=1e-2, heavy_tail=True)
        run.gpu_step()
        if step == 3:
            saved = [t.clone().cpu() for t in (run.buf.master, run.buf.m, run.buf.v, run.buf.scalars)]
    final = [t.clone().cpu() for t in (run.buf.master, run.buf.m, run.buf.v, run.buf.lp)]

    res = Job(psi, n_d, hp=hp, seed=7)
    for dst, src in zip((res.buf.master, res.buf.m, res.buf.v, res.buf.scalars), saved):
        dst.copy_(src.cuda())
    for step in range(4, 7):
        res.new_grads(step, sigma=1e-2, heavy_tail=True)
        res.gpu_step()
    again = [t.clone().cpu() for t in (res.buf.master, res.buf.m, res.buf.v, res.buf.lp)]
    for a, b in zip(final, again):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    assert res.scalars().t == 6


GUARD = 4096        # bytes of canary on each side of every buffer
CANARY = 0xA5


def _guarded(nbytes):
    """A device buffer with canary zones: returns (whole, inner view)."""
    whole = torch.full((GUARD + nbytes + GUARD,), CANARY, dtype=torch.uint8, device="cuda")
    return whole, whole[GUARD:GUARD + nbytes]


def _intact(whole):
    w = whole.cpu().numpy()
    return bool(np.all(w[:GUARD] == CANARY) and np.all(w[-GUARD:] == CANARY))


@pytest.mark.parametrize("n_d,psi,pad,clip,stage", [(4, 1_000_003, 8, 0.0, 2), (8, 123_457, 1, 1.0, 2),
                                                   (3, 70_001, 64, 0.0, 3), (16, 8193, 8, 1.0, 3)])
def test_no_kernel_writes_outside_its_buffers(n_d, psi, pad, clip, stage):
    hp = z.hparams(lr=1e-3, max_norm=clip)
    plan = z.Plan(psi, n_d, stage=stage, shard_pad=pad)
    n = plan.padded
    row = z.row_len(psi)
    bufs = {}
    for name, nbytes in (("grads", n_d * row * 2), ("master", 4 * n), ("m", 4 * n), ("v", 4 * n),
                         ("lp", 2 * (n if stage == 3 else psi)), ("ws", plan.workspace_bytes(hp)),
                         ("scalars", 256), ("gath", 2 * psi), ("g", 4 * n), ("codes", n),
                         ("scales", 4 * n_d * (-(-plan.shard // 2048))), ("qg", 2 * psi)):
        bufs[name] = _guarded(nbytes)
    inner = {k: v[1] for k, v in bufs.items()}
    grads = inner["grads"].view(torch.bfloat16).view(n_d, row)
    g = synth.rank_grads(n_d, psi, 1e-2, seed=3, step=1, row_pad=row - psi)
    grads.copy_(g.cuda())
    master, m, v = (inner[k].view(torch.float32) for k in ("master", "m", "v"))
    master.copy_(synth.master_init(n, psi, seed=3).cuda())
    m.zero_()
    v.zero_()
    sc = inner["scalars"]
    z.zero_scalars_init(sc)
    ranks = [grads[r] for r in range(n_d)]
    lp = inner["lp"].view(torch.bfloat16)
    for _ in range(2):
        z.zero_step_fused(plan.handle, hp, ranks, master, m, v, master, m, v, lp, sc, inner["ws"])
    gf = inner["g"].view(torch.float32)
    z.zero_reduce_scatter(plan.handle, ranks, hp, sc, gf, inner["ws"])
    z.zero_grad_sqnorm(plan.handle, None, hp, sc, inner["ws"])
    z.zero_adam_shard_step(plan.handle, hp, gf, master, m, v, lp, sc)
    S = plan.shard
    if stage == 3:
        z.zero_all_gather(plan.handle, [lp[r * S:(r + 1) * S] for r in range(n_d)],
                          inner["gath"].view(torch.bfloat16), sc)
    qsrc = lp if stage == 3 else inner["gath"].view(torch.bfloat16)
    if stage == 3:
        z.zero_quant_gather(plan.handle, qsrc, 2048, inner["codes"].view(torch.int8),
                            inner["scales"].view(torch.float32), inner["qg"].view(torch.bfloat16))
    if clip == 0.0:
        z.zero_step_fused_qgather(plan.handle, hp, ranks, master, m, v, master, m, v, 2048,
                                  inner["codes"].view(torch.int8), inner["scales"].view(torch.float32),
                                  inner["qg"].view(torch.bfloat16), sc, inner["ws"])
    torch.cuda.synchronize()
    for name, (whole, _) in bufs.items():
        assert _intact(whole), "a kernel wrote outside the %s buffer" % name
    assert z.read_scalars(sc).status == 0


def test_zero3_layerwise_loop_matches_the_oracle():
    # three layers of different sizes, N_d = 16: per step and per layer,
    # gather the layer's bf16 shards (the weights used by forward/backward),
    # then reduce-scatter + Adam writing the layer's bf16 shards
    n_d = 16
    sizes = [70_001, 4096 * 16 + 3, 123_457]
    hp = z.hparams(lr=1e-3)
    jobs = [Job(psi, n_d, stage=3, pad=8, hp=hp, seed=100 + i) for i, psi in enumerate(sizes)]
    for step in range(1, 4):
        for job in jobs:
            S = job.plan.shard
            gathered = torch.zeros(job.psi, dtype=torch.bfloat16, device="cuda")
            z.zero_all_gather(job.plan.handle, [job.buf.lp[r * S:(r + 1) * S] for r in range(n_d)], gathered,
                              job.buf.scalars)
            # the gathered weights are the oracle's previous shards, gathered
            want = oracle.all_gather_u16([job.o_lp_shards[r * S:(r + 1) * S] for r in range(n_d)], job.psi, S)
            assert np.array_equal(u16(gathered), want)
            job.new_grads(step)
            job.gpu_step()
            job.oracle_step()
            job.assert_bit_exact()


@pytest.mark.parametrize("n_d,psi,pad,clip", [(4, 1_000_003, 8, 0.0), (8, 123_457, 1, 1.0), (3, 70_001, 16, 0.0),
                                              (16, 8193, 8, 1.0), (5, 4097 * 3, 64, 0.0)])
def test_newer_kernels_write_only_their_buffers(n_d, psi, pad, clip):
    # the gradient sender (all ranks in one launch), the quantized-exchange
    # receiver, and gradient accumulation with the step at the last micro-batch
    hp = z.hparams(lr=1e-3, max_norm=clip)
    plan = z.Plan(psi, n_d, stage=2, shard_pad=pad)
    n, S = plan.padded, plan.shard
    row = z.row_len(psi)
    row16 = (psi + 15) // 16 * 16
    nbs = -(-S // 2048)
    n_dp = (n_d + 3) // 4 * 4
    sizes = {"grads": n_d * row * 2, "master": 4 * n, "m": 4 * n, "v": 4 * n, "lp": 2 * psi,
             "ws": plan.workspace_bytes(hp), "scalars": 256, "acc": 4 * n, "qscales": 4 * n_d * nbs * n_dp,
             "qscales256": 4 * n_d * -(-S // 256) * n_dp}
    for r in range(n_d):
        sizes["codes%d" % r] = row16
    bufs = {k: _guarded(v) for k, v in sizes.items()}
    inner = {k: v[1] for k, v in bufs.items()}
    grads = inner["grads"].view(torch.bfloat16).view(n_d, row)
    grads.copy_(synth.rank_grads(n_d, psi, 1e-2, seed=4, step=1, row_pad=row - psi).cuda())
    master, m, v = (inner[k].view(torch.float32) for k in ("master", "m", "v"))
    master.copy_(synth.master_init(n, psi, seed=4).cuda())
    m.zero_()
    v.zero_()
    sc = inner["scalars"]
    z.zero_scalars_init(sc)
    ranks = [grads[r] for r in range(n_d)]
    lp = inner["lp"].view(torch.bfloat16)
    acc = inner["acc"].view(torch.float32)
    codes = [inner["codes%d" % r].view(torch.int8) for r in range(n_d)]
    qscales = inner["qscales"].view(torch.float32)
    z.zero_accumulate_grads(plan.handle, ranks, None, acc, sc)
    z.zero_accumulate_grads(plan.handle, ranks, acc, acc, sc)
    z.zero_step_fused_accum(plan.handle, hp, ranks, acc, 3, master, m, v, master, m, v, lp, sc, inner["ws"])
    z.zero_quantize_grads(plan.handle, ranks, 2048, codes, qscales)
    z.zero_quantize_grads(plan.handle, ranks, 256, codes, inner["qscales256"].view(torch.float32))
    z.zero_quantize_grads(plan.handle, ranks, 2048, codes, qscales)
    if clip == 0.0:
        z.zero_step_fused_qgz(plan.handle, hp, codes, qscales, 2048, master, m, v, master, m, v, lp, sc)
    torch.cuda.synchronize()
    for name, (whole, _) in bufs.items():
        assert _intact(whole), "a kernel wrote outside the %s buffer" % name
    assert z.read_scalars(sc).status == 0
