"""GPU parity of the ZeRO-3 layer loop, zero_step_layers (itwiki "ZeRO-DP의
세 단계", "왜 통신량이 늘지 않는가": each layer's shards are all-gathered
before use and its gradients reduce-scattered; "DeepSpeed에서 쓰기":
overlap_comm / stage-3 prefetch).  Layers of different sizes, each with its
own stage-3 plan, one step-scalars block for the stack.  Every layer's
state and 16-bit shards must be the oracle's stage-3 step bit for bit, and
each gathered buffer the oracle's all-gather of the shards the step started
from -- whatever the schedule: all on one stream, or the gathers on a second
stream overlapping the steps, with one or two gathers per layer and as many
gathered buffers as layers or fewer."""
import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_02_gb300 as z
from gpu_helpers import Job, u16

pytestmark = pytest.mark.gpu

SIZES = [70_001, 4096 * 16 + 3, 123_457, 5, 40_000]


def _run(n_gathered, second_stream, gathers, n_d=8, steps=3):
    hp = z.hparams(lr=1e-3, weight_decay=0.01)
    jobs = [Job(psi, n_d, stage=3, pad=8, hp=hp, seed=200 + i) for i, psi in enumerate(SIZES)]
    scalars = torch.zeros(256, dtype=torch.uint8, device="cuda")
    z.zero_scalars_init(scalars)
    stack = z.LayerStack([(j.plan.handle, j.buf.rank_ptrs(), j.buf.master, j.buf.m, j.buf.v, j.buf.lp)
                          for j in jobs])
    size = max(SIZES)
    gathered = [torch.full((size,), 7.0, dtype=torch.bfloat16, device="cuda") for _ in range(n_gathered)]
    gs = torch.cuda.Stream() if second_stream else None
    for step in range(1, steps + 1):
        want = []
        for job in jobs:
            job.new_grads(step, sigma=1e-2, heavy_tail=True)
            S = job.plan.shard
            want.append(oracle.all_gather_u16([job.o_lp_shards[r * S:(r + 1) * S] for r in range(n_d)], job.psi, S))
        z.zero_step_layers(hp, stack, gathers, gathered, scalars, gather_stream=gs)
        torch.cuda.synchronize()
        sc = z.read_scalars(scalars)
        assert sc.t == step and sc.status == 0      # one commit for the whole stack
        for l, job in enumerate(jobs):
            # the buffer of layer l still holds it when no later layer shares it
            if l + n_gathered >= len(jobs):
                assert np.array_equal(u16(gathered[l % n_gathered][:job.psi]), want[l]), (step, l)
            job.oracle_step()
            job.assert_bit_exact()
    return jobs


@pytest.mark.parametrize("n_gathered,second_stream,gathers", [
    (len(SIZES), True, 1), (2, True, 1), (2, True, 2), (3, False, 1), (1, True, 1), (1, False, 2)])
def test_layer_loop_matches_the_oracle(n_gathered, second_stream, gathers):
    _run(n_gathered, second_stream, gathers)


def test_layer_loop_schedules_give_the_same_bits():
    a = _run(len(SIZES), True, 2, steps=2)
    b = _run(1, False, 1, steps=2)
    for x, y in zip(a, b):
        for t, u in ((x.buf.master, y.buf.master), (x.buf.m, y.buf.m), (x.buf.v, y.buf.v), (x.buf.lp, y.buf.lp)):
            assert torch.equal(t.view(torch.uint8), u.view(torch.uint8))


def test_layer_loop_work_is_done_when_the_calling_stream_is():
    # the call is made on a side stream; the gathers run on a third one: a
    # wait on the side stream alone must cover all of it
    n_d = 4
    hp = z.hparams(lr=1e-3)
    jobs = [Job(psi, n_d, stage=3, pad=8, hp=hp, seed=300 + i) for i, psi in enumerate((300_007, 200_003))]
    scalars = torch.zeros(256, dtype=torch.uint8, device="cuda")
    z.zero_scalars_init(scalars)
    gathered = [torch.zeros(300_007, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    for job in jobs:
        job.new_grads(1)
    torch.cuda.synchronize()
    side, gs = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(side):
        z.zero_step_layers(hp, [(j.plan.handle, j.buf.rank_ptrs(), j.buf.master, j.buf.m, j.buf.v, j.buf.lp)
                                for j in jobs], 2, gathered, scalars, stream=side, gather_stream=gs)
    side.synchronize()
    for job in jobs:
        S = job.plan.shard
        want = oracle.all_gather_u16([job.o_lp_shards[r * S:(r + 1) * S] for r in range(n_d)], job.psi, S)
        l = jobs.index(job)
        assert np.array_equal(u16(gathered[l][:job.psi]), want)
        job.oracle_step()
        job.assert_bit_exact()


def test_layer_loop_waits_for_each_layers_gradients():
    # each layer's gradients arrive on a side stream after a delay; its step
    # must wait for the layer's grads_ready event, and its stepped event must
    # cover the step (a copy of the shards ordered after it sees the update)
    n_d = 4
    hp = z.hparams(lr=1e-3)
    jobs = [Job(psi, n_d, stage=3, pad=8, hp=hp, seed=400 + i) for i, psi in enumerate((100_003, 60_001, 80_000))]
    scalars = torch.zeros(256, dtype=torch.uint8, device="cuda")
    z.zero_scalars_init(scalars)
    gathered = [torch.zeros(100_003, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    side, gs, out_s = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in jobs]
    stepped = [torch.cuda.Event() for _ in jobs]
    stack = z.LayerStack([(j.plan.handle, j.buf.rank_ptrs(), j.buf.master, j.buf.m, j.buf.v, j.buf.lp, ready[l],
                           stepped[l]) for l, j in enumerate(jobs)])
    for step in (1, 2):
        staged = []
        for job in jobs:
            g = job.new_grads(step)              # the oracle's rows; the device buffer is overwritten below
            staged.append(g.cuda())
            job.buf.grads.zero_()
        torch.cuda.synchronize()
        with torch.cuda.stream(side):
            for l, job in enumerate(jobs):
                torch.cuda._sleep(2_000_000)     # the "backward pass" of layer l
                job.buf.grads.copy_(staged[l])
                ready[l].record(side)
        z.zero_step_layers(hp, stack, 1, gathered, scalars, gather_stream=gs)
        snaps = []
        with torch.cuda.stream(out_s):
            for l, job in enumerate(jobs):
                out_s.wait_event(stepped[l])
                snaps.append(job.buf.lp.clone())
        out_s.synchronize()
        torch.cuda.synchronize()
        for l, job in enumerate(jobs):
            job.oracle_step()
            job.assert_bit_exact()
            assert np.array_equal(u16(snaps[l]), job.o_lp_shards)
