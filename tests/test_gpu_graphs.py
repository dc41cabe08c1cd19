"""The fused step captured into a CUDA graph (after one eager call on the
device, which caches the device attributes and kernel settings) replays with
the same bits as eager calls."""
import pytest
import torch

import zero_optimizer_step_02_gb300 as z
from zero_optimizer_step_02_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("hp_kw", [dict(lr=1e-3), dict(lr=3e-4, beta2=0.95, weight_decay=0.1, max_norm=1.0)])
def test_graph_replay_equals_eager(hp_kw):
    psi, n_d = 500_001, 8
    hp = z.hparams(**hp_kw)
    plan = z.Plan(psi, n_d, stage=2, shard_pad=8)
    jobs = []
    for _ in range(2):
        b = z.StepBuffers(plan, hp, device="cuda")
        b.master.copy_(synth.master_init(plan.padded, psi, seed=3, device="cuda"))
        b.grads.copy_(synth.rank_grads(n_d, psi, 1e-2, seed=5, step=1, device="cuda", heavy_tail=True,
                                       row_pad=b.grads.shape[1] - psi))
        b.init_scalars()
        b.step(hp)                                   # one eager call before any capture
        jobs.append(b)
    eager, graphed = jobs
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for _ in range(3):
                graphed.step(hp)
    torch.cuda.current_stream().wait_stream(stream)
    for _ in range(3):
        eager.step(hp)
    g.replay()
    torch.cuda.synchronize()
    for a, b in ((eager.master, graphed.master), (eager.m, graphed.m), (eager.v, graphed.v), (eager.lp, graphed.lp)):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    assert eager.scalars_host().t == graphed.scalars_host().t == 4
