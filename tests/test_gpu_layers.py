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
from gpu_helpers import ORACLE_DT, Job, _note_clipped_step, accum_ghat, coef_ulps, oracle_hp, step_with_coef, u16

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


# ----------------------------------------------- global checks across layers
def _global_step(jobs, hp, ghats, b1p, b2p, gpu_coef=None):
    """The oracle's view of one step of a stack that is one model: the clip
    norm over every layer's averaged gradient, in layer order (the oracle's
    sequential fp64 sum over the concatenation), one coefficient for all
    layers, each layer's Adam from its state before the step.  gpu_coef: the
    GPU's coefficient when it is one fp32 ulp from the oracle's (the norm is
    summed in another order), which the re-run then uses.  Returns the
    oracle's coefficient and squared norm; updates each job's oracle state
    and 16-bit shards."""
    ohp = oracle_hp(hp)
    coef, sq = np.float32(1.0), 0.0
    if hp.max_norm > 0:
        sq = oracle.sqnorm(np.concatenate([g[:j.psi] for g, j in zip(ghats, jobs)]))
        c, applied = oracle.clip_coef(hp.max_norm, sq)
        coef = np.float32(c) if applied else np.float32(1.0)
    use = coef if gpu_coef is None else np.float32(gpu_coef)
    for g, job in zip(ghats, jobs):
        st, lp = step_with_coef(job.ost, g, use, ohp, b1p, b2p, job.psi, ORACLE_DT[job.pdt])
        job.ost.master, job.ost.m, job.ost.v = st.master, st.m, st.v
        job.o_lp_shards[:job.psi] = lp
    return coef, sq


@pytest.mark.parametrize("n_d,second_stream,k", [(8, True, 1), (4, False, 1), (8, True, 2), (3, True, 3)])
def test_layer_loop_clips_by_the_norm_of_the_whole_stack(n_d, second_stream, k):
    # n_d = 8: the reduced gradients go through the workspace; n_d <= 4: the
    # update re-reads the ranks; k > 1: accumulated micro-batches
    hp = z.hparams(lr=3e-4, beta2=0.95, weight_decay=0.1, max_norm=1.0)
    sizes = (70_001, 4096 * 10 + 5, 30_000)
    jobs = [Job(psi, n_d, stage=3, pad=8, hp=hp, seed=500 + i) for i, psi in enumerate(sizes)]
    scalars = torch.zeros(256, dtype=torch.uint8, device="cuda")
    z.zero_scalars_init(scalars)
    layers = [(j.plan.handle, j.buf.rank_ptrs(), j.buf.master, j.buf.m, j.buf.v, j.buf.lp) for j in jobs]
    gathered = [torch.zeros(max(sizes), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    gs = torch.cuda.Stream() if second_stream else None
    b1p = b2p = 1.0
    taken = 0
    for step in range(1, 4):
        accs, ghats = [], []
        for job in jobs:
            acc = None
            for mu in range(1, k):
                job.new_grads(100 * step + mu, sigma=1e-2, heavy_tail=True)
                job.buf.accumulate(first=mu == 1)
                acc = oracle.accumulate_grads(job.rows, oracle.BF16, acc)
            job.new_grads(100 * step + k, sigma=1e-2, heavy_tail=True)
            accs.append(acc)
            job.snapshot()
            ghats.append(accum_ghat(job, acc, k))
        stack = z.LayerStack([l + (None, None, j.buf.acc if k > 1 else None) for l, j in zip(layers, jobs)])
        ws = torch.zeros(max(z.zero_layers_workspace_bytes(hp, stack), 256), dtype=torch.uint8, device="cuda")
        z.zero_step_layers(hp, stack, 1, gathered, scalars, ws=ws, micro_batches=k, gather_stream=gs)
        torch.cuda.synchronize()
        sc = z.read_scalars(scalars)
        assert sc.t == step and sc.status == 0
        b1p *= float(np.float32(hp.beta1))
        b2p *= float(np.float32(hp.beta2))
        coef, sq = _global_step(jobs, hp, ghats, b1p, b2p)
        assert coef < 1.0                                      # the clip is active
        psi_total = sum(sizes)
        assert sc.sqnorm == pytest.approx(sq, rel=2 * psi_total * 2.0 ** -53)
        d = coef_ulps(sc.clip_coef, coef)
        assert d <= 1
        _note_clipped_step(d == 1)
        if d == 1:
            taken += 1
            for job in jobs:
                job.ost = job.pre.copy()
            _global_step(jobs, hp, ghats, b1p, b2p, gpu_coef=sc.clip_coef)
        for job in jobs:
            job.assert_bit_exact()


@pytest.mark.parametrize("clip", [0.0, 1e-3])
def test_layer_loop_overflow_in_one_layer_skips_every_layer(clip):
    # fp16 gradients with a loss scale; at step 2 one layer holds +inf: no
    # layer changes, t stays, the scale halves
    n_d = 4
    hp = z.hparams(lr=1e-4, loss_scaling=True, max_norm=clip)
    sizes = (50_003, 20_000)
    jobs = [Job(psi, n_d, stage=3, pad=8, gdt=z.ZERO_FP16, hp=hp, seed=600 + i, loss_scale=1024.0)
            for i, psi in enumerate(sizes)]
    scalars = torch.zeros(256, dtype=torch.uint8, device="cuda")
    z.zero_scalars_init(scalars, 1024.0)
    stack = z.LayerStack([(j.plan.handle, j.buf.rank_ptrs(), j.buf.master, j.buf.m, j.buf.v, j.buf.lp) for j in jobs])
    ws = torch.zeros(max(z.zero_layers_workspace_bytes(hp, stack), 256), dtype=torch.uint8, device="cuda")
    gathered = [torch.zeros(max(sizes), dtype=torch.float16, device="cuda") for _ in range(2)]
    b1p = b2p = 1.0
    scale = 1024.0
    for step in range(1, 4):
        ghats = []
        for i, job in enumerate(jobs):
            inf_at = (1, 777) if (step == 2 and i == 1) else None
            job.new_grads(step, sigma=1e-4, scale=scale, inf_at=inf_at)
            ghats.append(oracle.reduce_scatter(job.rows, oracle.FP16, n_d * scale, job.plan.shard))
        before = [job.gpu_state() for job in jobs]
        z.zero_step_layers(hp, stack, 1, gathered, scalars, ws=ws, gather_stream=torch.cuda.Stream())
        torch.cuda.synchronize()
        sc = z.read_scalars(scalars)
        skipped = not all(np.all(np.isfinite(g[:j.psi])) for g, j in zip(ghats, jobs))
        assert skipped == (step == 2) and bool(sc.overflow) == skipped
        if skipped:
            scale /= 2
            for job, b in zip(jobs, before):
                for x, y in zip(b, job.gpu_state()):
                    assert np.array_equal(x, y)
        else:
            b1p *= float(np.float32(hp.beta1))
            b2p *= float(np.float32(hp.beta2))
            pre = [job.ost.copy() for job in jobs]
            coef, _ = _global_step(jobs, hp, ghats, b1p, b2p)
            if clip > 0:
                d = coef_ulps(sc.clip_coef, coef)
                assert coef < 1.0 and d <= 1
                _note_clipped_step(d == 1)
                if d == 1:
                    for job, p in zip(jobs, pre):
                        job.ost = p
                    _global_step(jobs, hp, ghats, b1p, b2p, gpu_coef=sc.clip_coef)
            for job in jobs:
                job.assert_bit_exact()
        assert sc.loss_scale == scale and sc.t == (step if step < 2 else step - 1)


@pytest.mark.parametrize("n_d,clip", [(8, 1.0), (4, 1.0), (8, 0.0)])
def test_layer_loop_with_state_in_host_memory(n_d, clip):
    # the itwiki DeepSpeed example offloads the optimizer state to the CPU:
    # layer 1 keeps master/m/v in page-locked host memory; the stack must give
    # the bits of the same stack with every state in HBM
    hp = z.hparams(lr=3e-4, beta2=0.95, weight_decay=0.1, max_norm=clip)
    sizes = (60_001, 4096 * 6 + 3)
    dev = [Job(psi, n_d, stage=3, pad=8, hp=hp, seed=700 + i) for i, psi in enumerate(sizes)]
    off = [Job(psi, n_d, stage=3, pad=8, hp=hp, seed=700 + i) for i, psi in enumerate(sizes)]
    hm, hmm, hv = (t.cpu().pin_memory() for t in (off[1].buf.master, off[1].buf.m, off[1].buf.v))
    gathered = [torch.zeros(max(sizes), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    sa, sb = (torch.zeros(256, dtype=torch.uint8, device="cuda") for _ in range(2))
    z.zero_scalars_init(sa)
    z.zero_scalars_init(sb)
    a = z.LayerStack([(j.plan.handle, j.buf.rank_ptrs(), j.buf.master, j.buf.m, j.buf.v, j.buf.lp) for j in dev])
    b = z.LayerStack([(off[0].plan.handle, off[0].buf.rank_ptrs(), off[0].buf.master, off[0].buf.m, off[0].buf.v,
                       off[0].buf.lp),
                      (off[1].plan.handle, off[1].buf.rank_ptrs(), hm, hmm, hv, off[1].buf.lp, None, None, None, True)])
    wa = torch.zeros(max(z.zero_layers_workspace_bytes(hp, a), 256), dtype=torch.uint8, device="cuda")
    wb = torch.zeros(max(z.zero_layers_workspace_bytes(hp, b), 256), dtype=torch.uint8, device="cuda")
    for step in (1, 2, 3):
        for x, y in zip(dev, off):
            x.new_grads(step, sigma=1e-2, heavy_tail=True)
            y.new_grads(step, sigma=1e-2, heavy_tail=True)
        z.zero_step_layers(hp, a, 1, gathered, sa, ws=wa, gather_stream=torch.cuda.Stream())
        z.zero_step_layers(hp, b, 1, gathered, sb, ws=wb, gather_stream=torch.cuda.Stream())
        torch.cuda.synchronize()
        for x, y, host in ((dev[0], off[0], None), (dev[1], off[1], (hm, hmm, hv))):
            ys = host if host else (y.buf.master, y.buf.m, y.buf.v)
            for t, u in zip((x.buf.master, x.buf.m, x.buf.v), ys):
                assert torch.equal(t.cpu().view(torch.int32), u.cpu().view(torch.int32))
            assert torch.equal(x.buf.lp.view(torch.int16), y.buf.lp.view(torch.int16))
        ra, rb = z.read_scalars(sa), z.read_scalars(sb)
        assert ra.t == rb.t == step and ra.sqnorm == rb.sqnorm and ra.status == rb.status == 0


@pytest.mark.parametrize("second_stream,gathers", [(True, 1), (False, 2)])
def test_layer_loop_with_quantized_gathers(second_stream, gathers):
    # ZeRO++ qwZ on the ZeRO-3 weight gathers (itwiki "후속 기법", ZeRO++ row):
    # each layer's gather block-quantizes its bf16 shards; codes, scales and
    # dequantized values bit for bit against the oracle's quantizer over the
    # shards the step started from; the steps themselves are unchanged
    n_d = 8
    hp = z.hparams(lr=1e-3, weight_decay=0.01)
    sizes = (70_001, 4096 * 9 + 7, 5)
    jobs = [Job(psi, n_d, stage=3, pad=8, hp=hp, seed=800 + i) for i, psi in enumerate(sizes)]
    scalars = torch.zeros(256, dtype=torch.uint8, device="cuda")
    z.zero_scalars_init(scalars)
    stack = z.LayerStack([(j.plan.handle, j.buf.rank_ptrs(), j.buf.master, j.buf.m, j.buf.v, j.buf.lp) for j in jobs])
    n_g = len(jobs)
    gathered = [torch.zeros(j.psi, dtype=torch.bfloat16, device="cuda") for j in jobs]
    codes = [torch.full((j.plan.padded,), 99, dtype=torch.int8, device="cuda") for j in jobs]
    scales = [torch.full((n_d * -(-j.plan.shard // 2048),), -1.0, device="cuda") for j in jobs]
    gs = torch.cuda.Stream() if second_stream else None
    for step in (1, 2, 3):
        want = []
        for job in jobs:
            job.new_grads(step, sigma=1e-2)
            want.append(oracle.quant_gather(job.o_lp_shards.copy(), n_d, job.psi, job.plan.shard, 2048))
        z.zero_step_layers(hp, stack, gathers, gathered, scalars, gather_stream=gs, gathered_codes=codes,
                           gathered_scales=scales)
        torch.cuda.synchronize()
        assert z.read_scalars(scalars).t == step
        for l, job in enumerate(jobs):
            oc, osc, og = want[l]
            assert np.array_equal(codes[l].cpu().numpy()[:job.psi], oc[:job.psi]), (step, l)
            assert np.array_equal(scales[l].cpu().numpy().view(np.uint32), osc.view(np.uint32)), (step, l)
            assert np.array_equal(u16(gathered[l]), og), (step, l)
            job.oracle_step()
            job.assert_bit_exact()
    assert n_g == len(gathered)
