"""Pins of the oracle's gradient accumulation (k micro-batches per step):
it reduces to the plain step at k = 1, its rounding order on a hand-worked
case, its mean over every micro-batch of every rank against plain data
parallelism on inputs whose sums are exact, and the loss-scaling skip."""
import numpy as np
import pytest

import oracle
from oracle import BF16, FP16


def _grads(n_d, psi, seed, sigma=1e-2, dtype=BF16, scale=1.0):
    rng = np.random.default_rng(seed)
    return [oracle.f32_to_lp((rng.normal(0, sigma, psi) * scale).astype(np.float32), dtype)
            for _ in range(n_d)]


def _grid_grads(n_d, psi, seed, dtype=BF16):
    # small integers times 2^-10: every rank and micro-batch sum below is exact
    rng = np.random.default_rng(seed)
    return [oracle.f32_to_lp((rng.integers(-100, 101, psi) * 2.0 ** -10).astype(np.float32), dtype)
            for _ in range(n_d)]


def _state(psi, n, seed, loss_scale=1.0):
    rng = np.random.default_rng(seed)
    master = np.zeros(n, np.float32)
    master[:psi] = rng.normal(0, 0.02, psi).astype(np.float32)
    return oracle.State(master, np.zeros(n, np.float32), np.zeros(n, np.float32), oracle.new_scalars(loss_scale))


def _bits(x):
    return np.asarray(x, np.float32).view(np.uint32)


@pytest.mark.parametrize("n_d,psi,pad,stage", [(1, 17, 8, 2), (4, 1003, 8, 2), (8, 4097, 64, 3), (3, 10, 1, 1)])
def test_one_micro_batch_is_the_plain_step(n_d, psi, pad, stage):
    hp = oracle.hparams(lr=3e-4, beta2=0.95, weight_decay=0.1, max_norm=0.05)
    S = oracle.shard_size(psi, n_d, pad)
    a, b = _state(psi, n_d * S, 1), _state(psi, n_d * S, 1)
    la, lb = np.zeros(n_d * S, np.uint16), np.zeros(n_d * S, np.uint16)
    ga, gb = np.zeros(psi, np.uint16), np.zeros(psi, np.uint16)
    for step in range(3):
        g = _grads(n_d, psi, seed=10 + step)
        oracle.zero_step(g, BF16, hp, a, pad, stage, lp_shards=la, gathered=ga)
        oracle.zero_step_accum(g, BF16, None, 1, hp, b, pad, stage, lp_shards=lb, gathered=gb)
        for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v)):
            assert np.array_equal(_bits(x), _bits(y))
        assert np.array_equal(la, lb) and np.array_equal(ga, gb)


def test_rounding_order_hand_worked():
    # Reading: each micro-batch's ranks are summed from +0 first, then the sum
    # is added to the accumulator.  Two elements, two ranks, two micro-batches
    # (all values exact in bf16), u = 2^-24 (half an ulp of 1.0 in fp32):
    #   element 0: micro 1 = (1, u), micro 2 = (0, u)
    #     micro 1: 1 + u is a tie, rounds to even: 1.0;  micro 2 sums to u;
    #     acc = 1 + u -> 1.0.  (Adding up each rank first would give
    #     (1 + 0) + (u + u) = 1 + 2^-23.)
    #   element 1: micro 1 = (1, 0), micro 2 = (u, u)
    #     micro 2 sums to 2u = 2^-23 exactly; acc = 1 + 2^-23, exact.
    #     (Continuing one running sum over all four values would give 1.0.)
    u = 2.0 ** -24
    m1 = [oracle.f32_to_bf16(np.array([1.0, 1.0], np.float32)), oracle.f32_to_bf16(np.array([u, 0.0], np.float32))]
    m2 = [oracle.f32_to_bf16(np.array([0.0, u], np.float32)), oracle.f32_to_bf16(np.array([u, u], np.float32))]
    acc = oracle.accumulate_grads(m1, BF16)
    acc = oracle.accumulate_grads(m2, BF16, acc)
    assert np.array_equal(_bits(acc), _bits([1.0, 1.0 + 2.0 ** -23]))


def test_first_micro_batch_starts_from_positive_zero():
    # -0 + -0 = -0 but +0 + -0 = +0: the sum starts from +0.0f
    g = [oracle.f32_to_bf16(np.array([-0.0, -0.0, 3.0], np.float32))] * 2
    acc = oracle.accumulate_grads(g, BF16)
    assert np.array_equal(_bits(acc), _bits([0.0, 0.0, 6.0]))
    # in place: acc_in and acc_out are one array element by element
    acc2 = oracle.accumulate_grads(g, BF16, acc)
    assert np.array_equal(_bits(acc2), _bits([0.0, 0.0, 12.0]))


@pytest.mark.parametrize("n_d,k,psi,pad,stage", [(2, 2, 1000, 8, 2), (4, 8, 257, 1, 3), (8, 3, 4097, 64, 2),
                                                 (1, 5, 33, 8, 1), (3, 4, 70, 16, 2)])
@pytest.mark.parametrize("variant", ["adam", "adamw_clip", "fp16_scaled"])
def test_mean_over_every_micro_batch_equals_plain_dp(n_d, k, psi, pad, stage, variant):
    # The effective batch of k micro-batches on n_d ranks is n_d * k rank
    # gradients: with every sum exact, the accumulated step must equal plain
    # data parallelism over n_d * k ranks (mean of all of them, one update).
    gdt = FP16 if variant == "fp16_scaled" else BF16
    scale = 256.0 if variant == "fp16_scaled" else 1.0
    hp = oracle.hparams(lr=3e-4 if variant == "adamw_clip" else 1e-3,
                        beta2=0.95 if variant == "adamw_clip" else 0.999,
                        weight_decay=0.1 if variant == "adamw_clip" else 0.0,
                        max_norm=0.05 if variant == "adamw_clip" else 0.0,
                        loss_scaling=variant == "fp16_scaled")
    S = oracle.shard_size(psi, n_d, pad)
    dp = _state(psi, psi, 5, scale)
    zs = _state(psi, n_d * S, 5, scale)
    zs.master[:psi] = dp.master[:psi]
    for step in range(2):
        micro = [_grid_grads(n_d, psi, seed=1000 * step + 10 * mu + n_d, dtype=gdt) for mu in range(k)]
        if scale != 1.0:
            micro = [[oracle.f32_to_lp(oracle.lp_to_f32(r, gdt) * np.float32(scale), gdt) for r in mb]
                     for mb in micro]
        acc = None
        for mu in range(k - 1):
            acc = oracle.accumulate_grads(micro[mu], gdt, acc)
        lp_sh, gath = np.zeros(n_d * S, np.uint16), np.zeros(psi, np.uint16)
        s1 = oracle.zero_step_accum(micro[-1], gdt, acc, k, hp, zs, pad, stage, lp_shards=lp_sh, gathered=gath)
        s2, lp_dp = oracle.plain_dp_step([r for mb in micro for r in mb], gdt, hp, dp)
        assert s1 == s2 == False
        for a, b in ((dp.master, zs.master), (dp.m, zs.m), (dp.v, zs.v)):
            assert np.array_equal(_bits(a[:psi]), _bits(b[:psi]))
        if stage == 3:
            for r in range(n_d):
                n = oracle.valid_len(psi, S, r)
                assert np.array_equal(lp_sh[r * S:r * S + n], lp_dp[r * S:r * S + n])
        else:
            assert np.array_equal(gath, lp_dp)
        assert zs.scalars.t == dp.scalars.t == step + 1


def test_accumulated_sum_against_exact_integers():
    # the accumulator holds the plain (undivided) sum of every micro-batch's
    # every rank gradient: on integer-valued inputs it is that integer
    rng = np.random.default_rng(4)
    n_d, k, psi = 5, 6, 300
    vals = rng.integers(-200, 201, size=(k, n_d, psi))
    acc = None
    for mu in range(k):
        acc = oracle.accumulate_grads([oracle.f32_to_bf16(vals[mu, r].astype(np.float32)) for r in range(n_d)], BF16,
                                      acc)
    assert np.array_equal(acc, vals.sum(axis=(0, 1)).astype(np.float32))


def test_overflow_in_an_early_micro_batch_skips_the_step():
    # fp16 loss scaling: an inf in micro-batch 1 stays non-finite in the
    # accumulator, so the step at micro-batch 3 is skipped and the scale halves
    n_d, psi, pad, k = 4, 200, 8, 3
    hp = oracle.hparams(loss_scaling=True, scale_window=100, min_scale=1.0)
    S = oracle.shard_size(psi, n_d, pad)
    st = _state(psi, n_d * S, 2, 1024.0)
    before = [a.copy() for a in (st.master, st.m, st.v)]
    micro = [_grads(n_d, psi, seed=mu, dtype=FP16, scale=1024.0) for mu in range(k)]
    micro[0][2][17] = np.uint16(0x7C00)   # +inf in fp16
    acc = oracle.accumulate_grads(micro[0], FP16)
    acc = oracle.accumulate_grads(micro[1], FP16, acc)
    assert np.isinf(acc[17])
    skipped = oracle.zero_step_accum(micro[2], FP16, acc, k, hp, st, pad, 2, gathered=np.zeros(psi, np.uint16))
    assert skipped
    assert st.scalars.t == 0 and st.scalars.loss_scale == 512.0
    for a, b in zip(before, (st.master, st.m, st.v)):
        assert np.array_equal(_bits(a), _bits(b))
