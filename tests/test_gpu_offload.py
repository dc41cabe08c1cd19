"""Optimizer state in page-locked host memory (ZeRO-Offload, GB300 style:
the GPU reads and writes the Grace-side state directly): the same bits as the
step with the state in HBM, under every pass schedule."""
import numpy as np
import pytest
import torch

import zero_optimizer_step_02_gb300 as z
from zero_optimizer_step_02_gb300 import synth

pytestmark = pytest.mark.gpu


def _host_state(n):
    return [torch.zeros(n, dtype=torch.float32).pin_memory() for _ in range(3)]


@pytest.mark.parametrize("n_d,psi,pad,hp_kw,pingpong", [
    (4, 1_000_003, 8, dict(lr=1e-3), False),                                     # one fused pass
    (8, 300_007, 8, dict(lr=3e-4, beta2=0.95, weight_decay=0.1, max_norm=1.0), False),  # reduce + Adam(g in HBM)
    (4, 300_007, 1, dict(lr=3e-4, weight_decay=0.1, max_norm=1.0), False),       # norm pass + fused
    (8, 200_003, 8, dict(lr=1e-4, loss_scaling=True), True),                     # speculative + repair
    (8, 200_003, 8, dict(lr=1e-4, loss_scaling=True), False),                    # check pass + guarded
])
def test_host_state_gives_the_device_bits(n_d, psi, pad, hp_kw, pingpong):
    hp = z.hparams(**hp_kw)
    ls = hp_kw.get("loss_scaling", False)
    gdt = z.ZERO_FP16 if ls else z.ZERO_BF16
    plan = z.Plan(psi, n_d, stage=2, grad_dtype=gdt, shard_pad=pad)
    n = plan.padded
    dev = z.StepBuffers(plan, hp, device="cuda", pingpong=pingpong)
    host_a, host_b = _host_state(n), _host_state(n)
    lp = torch.zeros(psi, dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(max(plan.workspace_bytes(hp), 256), dtype=torch.uint8, device="cuda")
    sc = torch.zeros(256, dtype=torch.uint8, device="cuda")
    master = synth.master_init(n, psi, seed=4)
    dev.master.copy_(master.cuda())
    host_a[0].copy_(master)
    scale = 1024.0 if ls else 1.0
    dev.init_scalars(scale)
    z.zero_scalars_init(sc, scale)
    cur, nxt = host_a, host_b
    for step in range(1, 5):
        g = synth.rank_grads(n_d, psi, 1e-4 if ls else 1e-2, seed=8, step=step, dtype=dev.grads.dtype,
                             scale=scale, row_pad=dev.grads.shape[1] - psi)
        if ls and step == 2:
            g[3, 777] = float("inf")
        dev.grads.copy_(g.cuda())
        dev.step(hp)
        outs = nxt if pingpong else cur
        z.zero_step_fused_offload(plan.handle, hp, dev.rank_list(), cur[0], cur[1], cur[2], outs[0], outs[1],
                                  outs[2], lp, sc, ws)
        if pingpong:
            cur, nxt = nxt, cur
        torch.cuda.synchronize()
        for a, b in zip((dev.master, dev.m, dev.v), cur):
            assert torch.equal(a.cpu().view(torch.int32), b.view(torch.int32))
        assert torch.equal(dev.lp[:psi].view(torch.int16), lp.view(torch.int16))
        s_dev, s_host = dev.scalars_host(), z.read_scalars(sc)
        assert (s_dev.t, s_dev.overflow, s_dev.loss_scale) == (s_host.t, s_host.overflow, s_host.loss_scale)
    if ls:
        assert z.read_scalars(sc).t == 3


def test_device_memory_is_refused_as_host_state():
    plan = z.Plan(10_000, 2, stage=2)
    hp = z.hparams()
    buf = z.StepBuffers(plan, hp, device="cuda")
    with pytest.raises(z.ZeroError) as e:
        z.zero_step_fused_offload(plan.handle, hp, buf.rank_list(), buf.master, buf.m, buf.v, buf.master, buf.m,
                                  buf.v, buf.lp, buf.scalars, buf.ws)
    assert e.value.status == 1
    pageable = torch.zeros(plan.padded)          # not page-locked
    with pytest.raises(z.ZeroError):
        z.zero_step_fused_offload(plan.handle, hp, buf.rank_list(), pageable, pageable, pageable, pageable, pageable,
                                  pageable, buf.lp, buf.scalars, buf.ws)
