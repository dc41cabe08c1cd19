"""The step's entry points captured into a CUDA graph (after one eager call
on the device, which caches the device attributes and kernel settings) replay
with the same bits as eager calls: the fused step, gradient accumulation, and
the quantized gradient exchange (sender and receiver; plain, clipped, and
with the int8 gather epilogue)."""
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


def _pair(psi, n_d, hp, stage=2):
    plan = z.Plan(psi, n_d, stage=stage, shard_pad=8)
    bufs = []
    for _ in range(2):
        b = z.StepBuffers(plan, hp, device="cuda")
        b.master.copy_(synth.master_init(plan.padded, psi, seed=3, device="cuda"))
        b.grads.copy_(synth.rank_grads(n_d, psi, 1e-2, seed=5, step=1, device="cuda",
                                       row_pad=b.grads.shape[1] - psi))
        b.init_scalars()
        bufs.append(b)
    return plan, bufs


def _capture(fn):
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            fn()
    torch.cuda.current_stream().wait_stream(stream)
    return g


def _same(a, b):
    for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v), (a.lp, b.lp)):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))


def test_accumulation_in_a_graph():
    # three micro-batches per step (two accumulations, then the step), twice
    hp = z.hparams(lr=1e-3, weight_decay=0.1, max_norm=1.0)
    plan, (eager, graphed) = _pair(300_007, 8, hp)

    def one_step(b):
        b.accumulate(first=True)
        b.accumulate(first=False)
        b.step_accum(hp, 3)

    for b in (eager, graphed):
        one_step(b)                                   # eager first calls
    g = _capture(lambda: [one_step(graphed) for _ in range(2)])
    for _ in range(2):
        one_step(eager)
    g.replay()
    torch.cuda.synchronize()
    _same(eager, graphed)
    assert torch.equal(eager.acc, graphed.acc)
    assert eager.scalars_host().t == graphed.scalars_host().t == 3


@pytest.mark.parametrize("mode", ["plain", "clip", "both", "both_clip"])
def test_quantized_exchange_in_a_graph(mode):
    # sender and receiver of the int8 gradient exchange, twice per graph;
    # clipped (reduce pass over the codes first) and with the int8 gather
    # epilogue of the two-exchange step
    hp = z.hparams(lr=1e-3, max_norm=1.0 if mode.endswith("clip") else 0.0)
    n_d, psi = 8, 300_007
    plan, (eager, graphed) = _pair(psi, n_d, hp)
    nbs = -(-plan.shard // 2048)
    wire, outs = [], []
    for _ in range(2):
        codes = torch.zeros(n_d, (psi + 15) // 16 * 16, dtype=torch.int8, device="cuda")
        scales = torch.zeros(n_d * nbs * ((n_d + 3) // 4 * 4), device="cuda")
        wire.append((codes, scales))
        outs.append((torch.zeros(plan.padded, dtype=torch.int8, device="cuda"),
                     torch.zeros(n_d * nbs, device="cuda"), torch.zeros(psi, dtype=torch.bfloat16, device="cuda")))

    def one_step(b, w, o):
        codes, scales = w
        rows = [codes[r] for r in range(n_d)]
        z.zero_quantize_grads(plan.handle, b.rank_list(), 2048, rows, scales, b.scalars)
        if mode.startswith("both"):
            z.zero_step_fused_qgz_qgather(plan.handle, hp, rows, scales, 2048, b.master, b.m, b.v, b.master, b.m,
                                          b.v, o[0], o[1], o[2], b.scalars, b.ws)
        else:
            z.zero_step_fused_qgz(plan.handle, hp, rows, scales, 2048, b.master, b.m, b.v, b.master, b.m, b.v,
                                  b.lp, b.scalars, b.ws)

    one_step(eager, wire[0], outs[0])
    one_step(graphed, wire[1], outs[1])
    g = _capture(lambda: [one_step(graphed, wire[1], outs[1]) for _ in range(2)])
    for _ in range(2):
        one_step(eager, wire[0], outs[0])
    g.replay()
    torch.cuda.synchronize()
    _same(eager, graphed)
    assert torch.equal(wire[0][0], wire[1][0]) and torch.equal(wire[0][1], wire[1][1])
    for x, y in zip(outs[0], outs[1]):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))
    se, sg = eager.scalars_host(), graphed.scalars_host()
    assert se.t == sg.t == 3 and se.clip_coef == sg.clip_coef
    if mode.endswith("clip"):
        assert se.clip_coef < 1.0
