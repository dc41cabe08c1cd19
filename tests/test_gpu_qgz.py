"""GPU parity of the quantized gradient exchange (ZeRO++ qgZ reading): the
sender's int8 codes and block scales, and the receiver's fused step (int8
codes dequantized, rank-ordered fp32 sum, Adam, cast), bit for bit against
the oracle on the same bytes."""
import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_02_gb300 as z
from gpu_helpers import oracle_hp, u16, u32
from zero_optimizer_step_02_gb300 import synth

pytestmark = pytest.mark.gpu


def _codes_buffers(n_d, psi, S, block):
    row = (psi + 15) // 16 * 16
    codes = torch.full((n_d, row), 77, dtype=torch.int8, device="cuda")
    nbs = -(-S // block)
    n_dp = (n_d + 3) // 4 * 4
    scales = torch.full((n_d * nbs * n_dp,), -1.0, device="cuda")
    return codes, scales, nbs


@pytest.mark.parametrize("n_d,psi,pad,block", [(2, 1 << 20, 8, 2048), (4, 1_000_003, 8, 2048),
                                               (3, 100_001, 1, 256), (8, 70_000, 64, 2048), (16, 5000, 8, 32),
                                               (1, 123_457, 8, 2048), (5, 4097 * 3, 1, 2048),
                                               (3, 100_001, 1, 2048), (64, 40_000, 16, 2048),
                                               (7, 6, 8, 2048), (2, 2 * 4096 * 37, 4096, 2048)])
def test_sender_codes_and_scales(n_d, psi, pad, block):
    plan = z.Plan(psi, n_d, stage=2, shard_pad=pad)
    S = plan.shard
    g = synth.rank_grads(n_d, psi, 1e-3, seed=5, step=1, row_pad=z.row_len(psi) - psi)
    gd = g.cuda()
    codes, scales, nbs = _codes_buffers(n_d, psi, S, block)
    z.zero_quantize_grads(plan.handle, [gd[r] for r in range(n_d)], block, [codes[r] for r in range(n_d)], scales)
    rows = [u16(g[r, :psi]) for r in range(n_d)]
    oc, osc = oracle.quantize_ranks(rows, psi, S, block)
    got_c = codes.cpu().numpy()
    got_s = scales.cpu().numpy().reshape(osc.shape)
    for q in range(n_d):
        assert np.array_equal(got_c[q, :psi], oc[q][:psi])
    assert np.array_equal(u32(got_s), u32(osc))         # rank padding columns included


@pytest.mark.parametrize("n_d,psi,pad", [(2, 1 << 20, 8), (4, 1_000_003, 16), (8, 123_457, 8), (3, 50_001, 1),
                                         (16, 300_007, 16), (64, 40_000, 16)])
@pytest.mark.parametrize("stage", [2, 3])
def test_receiver_fused_step(n_d, psi, pad, stage):
    hp = z.hparams(lr=1e-3, weight_decay=0.01)
    plan = z.Plan(psi, n_d, stage=stage, shard_pad=pad)
    S = plan.shard
    buf = z.StepBuffers(plan, hp, device="cuda")
    master = synth.master_init(plan.padded, psi, seed=9)
    buf.master.copy_(master.cuda())
    buf.init_scalars()
    st = oracle.State(master.numpy().copy(), np.zeros(plan.padded, np.float32), np.zeros(plan.padded, np.float32),
                      oracle.new_scalars())
    o_lp = np.zeros(plan.padded, np.uint16)
    o_g = np.zeros(psi, np.uint16)
    codes, scales, nbs = _codes_buffers(n_d, psi, S, 2048)
    for step in range(1, 4):
        g = synth.rank_grads(n_d, psi, 1e-3, seed=11, step=step, row_pad=z.row_len(psi) - psi)
        gd = g.cuda()
        z.zero_quantize_grads(plan.handle, [gd[r] for r in range(n_d)], 2048, [codes[r] for r in range(n_d)], scales)
        z.zero_step_fused_qgz(plan.handle, hp, [codes[r] for r in range(n_d)], scales, 2048, buf.master, buf.m,
                              buf.v, buf.master, buf.m, buf.v, buf.lp, buf.scalars)
        rows = [u16(g[r, :psi]) for r in range(n_d)]
        oc, osc = oracle.quantize_ranks(rows, psi, S, 2048)
        oracle.zero_step_qgz(oc, osc, 2048, oracle_hp(hp), st, pad, stage, psi, lp_shards=o_lp, gathered=o_g)
        torch.cuda.synchronize()
        for a, b in ((buf.master, st.master), (buf.m, st.m), (buf.v, st.v)):
            bad = np.flatnonzero(u32(a.cpu().numpy()) != u32(b))
            assert bad.size == 0, "%d elements differ, first %s" % (bad.size, bad[:5])
        want_lp = o_lp[:psi] if stage == 3 else o_g
        assert np.array_equal(u16(buf.lp[:psi]), want_lp)
        sc = buf.scalars_host()
        assert sc.t == step and sc.status == 0


def test_receiver_on_grid_equals_the_plain_fused_step():
    # gradients on the int8 grid (every block's max is 127 * 2^-10): the
    # quantized exchange is lossless and must give the plain step's bits
    n_d, psi, pad = 4, 4096 * 40, 16
    plan = z.Plan(psi, n_d, stage=2, shard_pad=pad)
    S = plan.shard
    hp = z.hparams(lr=1e-3)
    rng = np.random.default_rng(0)
    k = rng.integers(-127, 128, size=(n_d, psi)).astype(np.float32)
    k[:, ::2048] = 127.0
    x = torch.from_numpy(k * 2.0 ** -10).to(torch.bfloat16)
    grads = torch.zeros(n_d, z.row_len(psi), dtype=torch.bfloat16)
    grads[:, :psi] = x
    a = z.StepBuffers(plan, hp, device="cuda", grads=grads.cuda())
    b = z.StepBuffers(plan, hp, device="cuda")
    master = synth.master_init(plan.padded, psi, seed=1, device="cuda")
    for s in (a, b):
        s.master.copy_(master)
        s.init_scalars()
    codes, scales, _ = _codes_buffers(n_d, psi, S, 2048)
    z.zero_quantize_grads(plan.handle, a.rank_list(), 2048, [codes[r] for r in range(n_d)], scales)
    a.step(hp)
    z.zero_step_fused_qgz(plan.handle, hp, [codes[r] for r in range(n_d)], scales, 2048, b.master, b.m, b.v,
                          b.master, b.m, b.v, b.lp, b.scalars)
    torch.cuda.synchronize()
    assert torch.equal(a.master.view(torch.int32), b.master.view(torch.int32))
    assert torch.equal(a.lp.view(torch.int16), b.lp.view(torch.int16))


@pytest.mark.parametrize("n_d,psi,pad", [(3, 50_001, 1), (16, 200_003, 16), (17, 70_001, 8), (64, 300_000, 16)])
def test_receiver_decodes_every_byte(n_d, psi, pad):
    # codes drawn over all 256 byte values (the sender never writes -128, but
    # the receiver takes any int8 as its value) with random positive and zero
    # scales: the decode of each byte and each scale product, bit for bit
    hp = z.hparams(lr=1e-3)
    plan = z.Plan(psi, n_d, stage=2, shard_pad=pad)
    S = plan.shard
    buf = z.StepBuffers(plan, hp, device="cuda")
    master = synth.master_init(plan.padded, psi, seed=3)
    buf.master.copy_(master.cuda())
    buf.init_scalars()
    st = oracle.State(master.numpy().copy(), np.zeros(plan.padded, np.float32), np.zeros(plan.padded, np.float32),
                      oracle.new_scalars())
    o_g = np.zeros(psi, np.uint16)
    codes, scales, nbs = _codes_buffers(n_d, psi, S, 2048)
    rng = np.random.default_rng(n_d * 1000 + psi)
    oc = [rng.integers(-128, 128, size=psi).astype(np.int8) for _ in range(n_d)]
    oc[0][:256] = np.arange(-128, 128, dtype=np.int8)
    n_dp = oracle.qgz_rank_stride(n_d)
    osc = np.zeros((n_d * nbs, n_dp), np.float32)
    osc[:, :n_d] = np.exp(rng.uniform(-14.0, -6.0, size=(n_d * nbs, n_d))).astype(np.float32)
    osc[:, :n_d][rng.random((n_d * nbs, n_d)) < 0.05] = 0.0
    for q in range(n_d):
        codes[q, :psi] = torch.from_numpy(oc[q]).cuda()
    scales.copy_(torch.from_numpy(osc.reshape(-1)).cuda())
    z.zero_step_fused_qgz(plan.handle, hp, [codes[r] for r in range(n_d)], scales, 2048, buf.master, buf.m, buf.v,
                          buf.master, buf.m, buf.v, buf.lp, buf.scalars)
    oracle.zero_step_qgz(oc, osc, 2048, oracle_hp(hp), st, pad, 2, psi, gathered=o_g)
    torch.cuda.synchronize()
    for a, b in ((buf.master, st.master), (buf.m, st.m), (buf.v, st.v)):
        bad = np.flatnonzero(u32(a.cpu().numpy()) != u32(b))
        assert bad.size == 0, "%d elements differ, first %s" % (bad.size, bad[:5])
    assert np.array_equal(u16(buf.lp[:psi]), o_g)
    assert buf.scalars_host().status == 0
