"""Pins of the oracle's full step: ZeRO equals plain data parallelism bit for
bit (the pages' invariant), the clipping rule against closed forms, the
overflow skip against a run that never saw the bad step, and the block
quantizer against its defining properties."""
import itertools

import numpy as np
import pytest

import oracle
from oracle import BF16, FP16


def _grads(n_d, psi, seed, sigma=1e-3, dtype=BF16, scale=1.0):
    rng = np.random.default_rng(seed)
    return [oracle.f32_to_lp((rng.normal(0, sigma, psi) * scale).astype(np.float32), dtype)
            for _ in range(n_d)]


def _state(psi, n, seed):
    rng = np.random.default_rng(seed)
    master = np.zeros(n, np.float32)
    master[:psi] = rng.normal(0, 0.02, psi).astype(np.float32)
    return oracle.State(master, np.zeros(n, np.float32), np.zeros(n, np.float32),
                        oracle.new_scalars(1.0))


CASES = [(1, 1, 1), (1, 17, 8), (2, 1, 1), (2, 9, 1), (3, 1000, 8), (4, 1003, 8), (4, 3, 1),
         (5, 4, 64), (8, 7, 8), (8, 4097, 64), (16, 1000, 8), (64, 63, 1), (64, 5000, 8)]


@pytest.mark.parametrize("n_d,psi,pad", CASES)
@pytest.mark.parametrize("stage", [1, 2, 3])
@pytest.mark.parametrize("variant", ["adam", "adamw_clip", "fp16_scaled"])
def test_zero_step_equals_plain_dp_step(n_d, psi, pad, stage, variant):
    # "Data parallelism and ZeRO optimization", ZeRO-1: a parameter's optimizer
    # state depends only on its own gradient, so each rank may update its own
    # partition; "大模型并行技术": ZeRO is data parallelism in essence.  Hence the
    # ZeRO step must reproduce the plain all-reduce -> update -> replicate step.
    gdt = FP16 if variant == "fp16_scaled" else BF16
    hp = oracle.hparams(lr=3e-4 if variant == "adamw_clip" else 1e-3,
                        beta2=0.95 if variant == "adamw_clip" else 0.999,
                        weight_decay=0.1 if variant == "adamw_clip" else 0.0,
                        max_norm=0.05 if variant == "adamw_clip" else 0.0,
                        loss_scaling=variant == "fp16_scaled")
    S = oracle.shard_size(psi, n_d, pad)
    dp = _state(psi, psi, seed=psi)
    zs = _state(psi, n_d * S, seed=psi)
    zs.master[:psi] = dp.master
    scale = 1024.0 if variant == "fp16_scaled" else 1.0
    dp.scalars.loss_scale = zs.scalars.loss_scale = scale
    for step in range(3):
        g = _grads(n_d, psi, seed=100 * step + n_d, sigma=1e-2, dtype=gdt, scale=scale)
        s1, lp_dp = oracle.plain_dp_step(g, gdt, hp, dp)
        lp_sh = np.zeros(n_d * S, np.uint16)
        gath = np.zeros(psi, np.uint16)
        s2 = oracle.zero_step(g, gdt, hp, zs, pad, stage, lp_shards=lp_sh, gathered=gath)
        assert s1 == s2 == False
        for a, b in ((dp.master, zs.master), (dp.m, zs.m), (dp.v, zs.v)):
            assert np.array_equal(a.view(np.uint32), b[:psi].view(np.uint32))
            assert not b[psi:].view(np.uint32).any()          # padding stays +0
        got_lp = lp_sh[:psi] if stage == 3 else gath
        assert np.array_equal(lp_dp, got_lp)
        assert dp.scalars.t == zs.scalars.t == step + 1
        assert dp.scalars.sqnorm == zs.scalars.sqnorm
        assert dp.scalars.clip_coef == zs.scalars.clip_coef
        if stage == 3:
            assert not lp_sh[psi:].any()


def test_clip_coefficient_closed_form():
    # every averaged gradient entry is c = 2^-3 over psi = 4096 entries:
    # norm = |c| sqrt(psi) = 8 exactly, coef = max_norm / (8 + 1e-6)
    psi, n_d = 4096, 4
    g = [oracle.f32_to_bf16(np.full(psi, 0.125, np.float32))] * n_d
    st = _state(psi, psi, 0)
    hp = oracle.hparams(max_norm=1.0)
    oracle.plain_dp_step(g, BF16, hp, st)
    assert st.scalars.sqnorm == 64.0
    assert st.scalars.clip_coef == np.float32(1.0 / (8.0 + 1e-6))
    # after clipping the gradient norm is max_norm (to fp32 rounding)
    clipped = np.float32(0.125) * np.float32(st.scalars.clip_coef)
    assert np.sqrt(psi) * float(clipped) == pytest.approx(1.0, rel=1e-6)


def test_clip_not_applied_below_threshold_and_infinite_max_norm():
    psi, n_d = 1000, 2
    g = _grads(n_d, psi, 7, sigma=1e-3)
    base = _state(psi, psi, 1)
    a, b, c = base.copy(), base.copy(), base.copy()
    oracle.plain_dp_step(g, BF16, oracle.hparams(), a)
    oracle.plain_dp_step(g, BF16, oracle.hparams(max_norm=float("inf")), b)
    oracle.plain_dp_step(g, BF16, oracle.hparams(max_norm=1e6), c)
    for x in (b, c):
        assert np.array_equal(a.master, x.master) and np.array_equal(a.v, x.v)
        assert x.scalars.clip_coef == 1.0


def test_clip_scales_the_gradient_linearly():
    # a clipped step with gradient G equals an unclipped step with coef * G when
    # coef * G is exact (power-of-two coef): choose the norm so coef = 1/2.
    psi, n_d = 256, 1
    # one entry 2^-1, rest zero: norm = 0.5; max_norm = 0.25 (1 + 2e-6) -> coef = 0.5 in fp32
    x = np.zeros(psi, np.float32)
    x[3] = 0.5
    g = [oracle.f32_to_bf16(x)]
    max_norm = float(np.float32(0.25 * (1 + 2e-6)))
    a, b = _state(psi, psi, 2), _state(psi, psi, 2)
    oracle.plain_dp_step(g, BF16, oracle.hparams(max_norm=max_norm), a)
    assert a.scalars.clip_coef == 0.5
    oracle.plain_dp_step([oracle.f32_to_bf16(x * 0.5)], BF16, oracle.hparams(), b)
    assert np.array_equal(a.master, b.master) and np.array_equal(a.m, b.m)


@pytest.mark.parametrize("bad", [np.inf, -np.inf, np.nan])
@pytest.mark.parametrize("stage", [1, 2, 3])
def test_overflow_skip_equals_a_run_without_the_bad_step(bad, stage):
    # loss scaling (a reading; not on the pages): the step with a non-finite
    # gradient is skipped, state untouched, scale halved, t not advanced.
    n_d, psi, pad = 8, 3001, 8
    S = oracle.shard_size(psi, n_d, pad)
    hp = oracle.hparams(lr=1e-4, loss_scaling=True)
    run = _state(psi, n_d * S, 3)
    ref = run.copy()
    run.scalars.loss_scale = ref.scalars.loss_scale = 1024.0
    buf = dict(lp_shards=np.zeros(n_d * S, np.uint16), gathered=np.zeros(psi, np.uint16))
    for step in range(1, 7):
        scale = run.scalars.loss_scale
        g = _grads(n_d, psi, 50 + step, sigma=1e-4, dtype=FP16, scale=scale)
        if step == 3:
            g[5] = g[5].copy()
            g[5][1234] = oracle.f32_to_fp16(np.array([bad], np.float32))[0]
            before = run.copy()
            assert oracle.zero_step(g, FP16, hp, run, pad, stage, **buf)
            assert run.scalars.overflow == 1 and run.scalars.t == 2
            assert run.scalars.loss_scale == 512.0 and run.scalars.good_steps == 0
            for a, b in ((before.master, run.master), (before.m, run.m), (before.v, run.v)):
                assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
            ref.scalars.loss_scale = 512.0
            ref.scalars.good_steps = 0
            continue
        assert not oracle.zero_step(g, FP16, hp, run, pad, stage, **buf)
        assert not oracle.zero_step(g, FP16, hp, ref, pad, stage, **buf)
        assert np.array_equal(run.master, ref.master) and np.array_equal(run.v, ref.v)
    assert run.scalars.t == 5


def test_loss_scale_floor_and_growth():
    psi, n_d = 64, 2
    hp = oracle.hparams(loss_scaling=True, scale_window=2, min_scale=1.0)
    st = _state(psi, psi, 4)
    st.scalars.loss_scale = 2.0
    bad = _grads(n_d, psi, 1, dtype=FP16)
    bad[0] = bad[0].copy()
    bad[0][0] = 0x7C00
    for want in (1.0, 1.0):
        assert oracle.plain_dp_step(bad, FP16, hp, st)[0]
        assert st.scalars.loss_scale == want
    good = _grads(n_d, psi, 2, dtype=FP16)
    oracle.plain_dp_step(good, FP16, hp, st)
    assert st.scalars.loss_scale == 1.0 and st.scalars.good_steps == 1
    oracle.plain_dp_step(good, FP16, hp, st)
    assert st.scalars.loss_scale == 2.0 and st.scalars.good_steps == 0


def test_without_loss_scaling_nonfinite_propagates():
    psi, n_d = 16, 2
    g = _grads(n_d, psi, 3)
    g[1] = g[1].copy()
    g[1][4] = 0x7F80  # bf16 +inf
    st = _state(psi, psi, 5)
    skipped, _ = oracle.plain_dp_step(g, BF16, oracle.hparams(), st)
    assert not skipped and st.scalars.t == 1
    assert not np.isfinite(st.v[4])


# ------------------------------------------------------------- quantizer --
def _bf16(x):
    return oracle.f32_to_bf16(np.asarray(x, np.float32))


@pytest.mark.parametrize("seed", range(4))
def test_quantizer_properties(seed):
    rng = np.random.default_rng(seed)
    x = _bf16(rng.normal(0, 0.02, 2048) * (10.0 ** rng.uniform(-3, 1)))
    codes, s, deq = oracle.quantize_block(x)
    xf = oracle.bf16_to_f32(x).astype(np.float64)
    amax = np.abs(xf).max()
    assert s == np.float32(np.float32(amax) / np.float32(127.0))
    assert np.abs(codes).max() == 127
    assert np.abs(codes[np.argmax(np.abs(xf))]) == 127
    assert np.all(np.sign(codes[codes != 0]) == np.sign(xf[codes != 0]))
    # rounding to nearest: |x/s - q| <= 1/2 plus the rounding of the fp32
    # quotient x/s itself (half an ulp of a value below 128: 2^-17)
    assert np.all(np.abs(xf - codes.astype(np.float64) * s) <= s * (0.5 + 2.0 ** -17))
    # the dequantized value is the bf16 of q * s
    assert np.array_equal(deq, _bf16(codes.astype(np.float32) * np.float32(s)))


def test_quantizer_zero_block_and_grid_round_trip():
    codes, s, deq = oracle.quantize_block(_bf16(np.zeros(2048)))
    assert s == 0.0 and not codes.any() and not deq.any()
    k = np.arange(-127, 128)
    x = _bf16(k * 2.0 ** -10)        # amax = 127 * 2^-10 -> s = 2^-10 exactly
    codes, s, deq = oracle.quantize_block(x)
    assert s == 2.0 ** -10
    assert np.array_equal(codes, k.astype(np.int8)) and np.array_equal(deq, x)


def test_quantizer_ties_to_even():
    # s = 2^-10; 2.5 s -> 2, 3.5 s -> 4, -2.5 s -> -2
    x = _bf16(np.array([127, 2.5, 3.5, -2.5, 0.5, 1.5]) * 2.0 ** -10)
    codes, s, _ = oracle.quantize_block(x)
    assert list(codes) == [127, 2, 4, -2, 0, 2]


def test_quantizer_non_finite_weights():
    # clamp(q) = min(max(q, -127), 127) with IEEE maxNum / minNum, which return
    # the other operand when one is NaN: a NaN quotient has code -127.  The
    # absmax skips a NaN (max |x| over the numbers), so a NaN weight in a
    # finite block gets -127 and dequantizes to -127 s; an infinite weight
    # makes s infinite, so the finite weights' quotients are 0 and the
    # infinite one's is inf / inf = NaN
    s_want = np.float32(np.float32(2.0) / np.float32(127.0))
    codes, s, deq = oracle.quantize_block(_bf16([1.0, np.nan, -2.0, 0.0]))
    assert s == s_want
    assert list(codes) == [64, -127, -127, 0]     # 1 / (2/127) = 63.5 -> 64 (ties to even)
    assert np.array_equal(deq, _bf16(np.array([64, -127, -127, 0], np.float32) * s_want))
    codes, s, deq = oracle.quantize_block(_bf16([1.0, np.inf, -3.0, np.nan]))
    assert s == np.inf
    assert list(codes) == [0, -127, 0, -127]
    d = oracle.bf16_to_f32(deq)
    assert np.isnan(d[0]) and d[1] == -np.inf and np.isnan(d[2]) and d[3] == -np.inf   # 0 * inf, -127 * inf


@pytest.mark.parametrize("n_d,psi,pad,block", [(2, 5000, 8, 2048), (4, 1003, 1, 256),
                                               (3, 7000, 64, 2048), (8, 100, 8, 32)])
def test_quant_gather_blocks_follow_shards(n_d, psi, pad, block):
    S = oracle.shard_size(psi, n_d, pad)
    rng = np.random.default_rng(psi)
    flat = np.zeros(n_d * S, np.uint16)
    flat[:psi] = _bf16(rng.normal(0, 0.02, psi))
    codes, scales, gathered = oracle.quant_gather(flat, n_d, psi, S, block)
    nbs = -(-S // block)
    for r in range(n_d):
        L = oracle.valid_len(psi, S, r)
        for b in range(nbs):
            lo, hi = b * block, min((b + 1) * block, L)
            if hi <= lo:
                assert scales[r * nbs + b] == 0.0
                continue
            c, s, d = oracle.quantize_block(flat[r * S + lo:r * S + hi])
            assert scales[r * nbs + b] == s
            assert np.array_equal(codes[r * S + lo:r * S + hi], c)
            assert np.array_equal(gathered[r * S + lo:r * S + hi], d)


@pytest.mark.parametrize("wd", [0.0, 0.1])
def test_full_steps_follow_textbook_adam(wd):
    # one rank, so the averaged gradient is exactly the widened input; five full
    # steps through the step bookkeeping (beta powers, t) against textbook AdamW
    # in 50-digit decimals, and beta^t against its decimal value
    from decimal import Decimal
    from test_oracle_adam import _textbook
    psi = 5
    hp = oracle.hparams(lr=1e-2, beta1=0.9, beta2=0.99, weight_decay=wd)
    st = _state(psi, psi, 9)
    p0 = st.master.copy()
    gs = []
    for step in range(5):
        g = _grads(1, psi, 300 + step, sigma=0.1)
        gs.append(oracle.bf16_to_f32(g[0]))
        oracle.plain_dp_step(g, BF16, hp, st)
    tp, tm, tv = _textbook(hp, p0, gs, wd)
    assert np.allclose(st.m, tm, rtol=1e-5) and np.allclose(st.v, tv, rtol=1e-5)
    assert np.allclose(st.master, tp, rtol=0, atol=1e-6)
    assert st.scalars.t == 5
    b1, b2 = Decimal(float(np.float32(0.9))), Decimal(float(np.float32(0.99)))
    assert st.scalars.beta1_pow == pytest.approx(float(b1 ** 5), rel=1e-15)
    assert st.scalars.beta2_pow == pytest.approx(float(b2 ** 5), rel=1e-15)


@pytest.mark.parametrize("n_d", [1, 2, 8])
def test_loss_scale_divides_out(n_d):
    # fp16 gradients that are exact multiples of the scale: a loss-scaled step
    # on G * 1024 must equal an unscaled step on G (both exact in fp16)
    psi = 777
    rng = np.random.default_rng(n_d)
    G = [np.round(rng.normal(0, 8, psi)).astype(np.float32) / 64 for _ in range(n_d)]
    scaled = [oracle.f32_to_fp16(x * 1024) for x in G]
    plain = [oracle.f32_to_fp16(x) for x in G]
    a, b = _state(psi, psi, 11), _state(psi, psi, 11)
    a.scalars.loss_scale = 1024.0
    oracle.plain_dp_step(scaled, FP16, oracle.hparams(loss_scaling=True), a)
    oracle.plain_dp_step(plain, FP16, oracle.hparams(), b)
    assert np.array_equal(a.master, b.master) and np.array_equal(a.v, b.v)
