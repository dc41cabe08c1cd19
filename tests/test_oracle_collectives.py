"""Pins of the oracle's partition and collectives: the layout by the
properties that define it, reduce-scatter then all-gather equal to
all-reduce, and hand-computed sums where the rank order and the fp32
rounding decide the result."""
import itertools

import numpy as np
import pytest
import torch

import oracle
from oracle import BF16, FP16


def _bf16(vals):
    return oracle.f32_to_bf16(np.asarray(vals, dtype=np.float32))


def _rand_grads(n_d, psi, seed, sigma=1e-3, dtype=BF16):
    rng = np.random.default_rng(seed)
    return [oracle.f32_to_lp(rng.normal(0, sigma, psi).astype(np.float32), dtype) for _ in range(n_d)]


@pytest.mark.parametrize("psi", [0, 1, 2, 3, 7, 8, 63, 64, 65, 100, 1000, 1003])
@pytest.mark.parametrize("n_d", [1, 2, 3, 4, 5, 8, 16, 64])
@pytest.mark.parametrize("pad", [1, 2, 8, 64])
def test_layout_is_the_minimal_padded_contiguous_split(psi, n_d, pad):
    # "Data parallelism and ZeRO optimization", ZeRO-1: theta = [theta_1 .. theta_N],
    # rank r owns theta_r.  The reading: equal contiguous rank-ordered shards of
    # size S, a multiple of the pad, S the smallest such size with n_d * S >= psi.
    S = oracle.shard_size(psi, n_d, pad)
    assert S % pad == 0 and n_d * S >= psi
    assert S == 0 or n_d * (S - pad) < psi
    lens = [oracle.valid_len(psi, S, r) for r in range(n_d)]
    assert sum(lens) == psi
    covered = []
    for r, L in enumerate(lens):
        assert 0 <= L <= S
        if L:
            covered.extend(range(r * S, r * S + L))
    assert covered == list(range(psi))
    # only the trailing shards are short, and after the first short one all are empty
    short = [r for r, L in enumerate(lens) if L < S]
    if short:
        assert all(lens[r] == 0 for r in short[1:])
    for j in range(psi):
        r, i = oracle.owner(j, S)
        assert r * S + i == j and i < lens[r]


def test_small_workload_shard_layout():
    # Psi = 1,000,003 over 4 ranks: pad 8 -> S = 250,008; pad 1 -> S = 250,001
    S = oracle.shard_size(1_000_003, 4, 8)
    assert S == 250_008 and oracle.valid_len(1_000_003, S, 3) == 249_979
    S1 = oracle.shard_size(1_000_003, 4, 1)
    assert S1 == 250_001 and oracle.valid_len(1_000_003, S1, 3) == 250_000


@pytest.mark.parametrize("n_d,psi,pad", [(1, 5, 1), (2, 9, 1), (3, 1000, 8), (4, 1_003, 64),
                                         (8, 7, 8), (16, 4097, 8), (64, 333, 1)])
@pytest.mark.parametrize("dtype", [BF16, FP16])
def test_reduce_scatter_then_all_gather_is_all_reduce(n_d, psi, pad, dtype):
    # "ZeRO (딥 러닝)", 왜 통신량이 늘지 않는가: all-reduce = reduce-scatter + all-gather
    grads = _rand_grads(n_d, psi, seed=n_d * 1000 + psi, dtype=dtype)
    S = oracle.shard_size(psi, n_d, pad)
    D = float(n_d)
    rs = oracle.reduce_scatter(grads, dtype, D, S)
    ag = oracle.all_gather_f32([rs[r * S:(r + 1) * S] for r in range(n_d)], psi, S)
    ar = oracle.all_reduce_mean(grads, dtype, D)
    assert np.array_equal(ag.view(np.uint32), ar.view(np.uint32))
    # padding of the reduce-scatter output is +0
    mask = np.ones(n_d * S, dtype=bool)
    for r in range(n_d):
        mask[r * S:r * S + oracle.valid_len(psi, S, r)] = False
    assert np.all(rs[mask].view(np.uint32) == 0)


@pytest.mark.parametrize("n_d", [1, 2, 3, 5, 7, 8, 64])
def test_identical_ranks_average_to_the_value(n_d):
    # sum of n equal bf16 values is exact in fp32, so the mean is the value itself
    x = _bf16(np.random.default_rng(n_d).normal(0, 1, 257))
    ar = oracle.all_reduce_mean([x] * n_d, BF16, float(n_d))
    assert np.array_equal(oracle.f32_to_bf16(ar), x)


def test_single_rank_is_the_widening_cast():
    x = _bf16(np.random.default_rng(5).normal(0, 1, 1001))
    want = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    assert np.array_equal(oracle.all_reduce_mean([x], BF16, 1.0), want)


def test_rank_order_decides_the_rounding():
    # ranks 0..2 hold 1, 2^-24, 2^-24.  In rank order: (1 + 2^-24) ties to 1, then
    # again 1, so the mean is fl(1/3).  Any other order that adds the two small
    # values first gives 1 + 2^-23 instead.
    g = [_bf16([1.0]), _bf16([2.0 ** -24]), _bf16([2.0 ** -24])]
    got = oracle.all_reduce_mean(g, BF16, 3.0)[0]
    assert got == np.float32(1.0) / np.float32(3.0)
    rev = oracle.all_reduce_mean(g[::-1], BF16, 3.0)[0]
    assert rev == np.float32(1.0 + 2.0 ** -23) / np.float32(3.0)
    assert got != rev


def test_mean_divides_by_rank_count_and_loss_scale():
    # two ranks, 3.0 and 5.0, loss scale 1024: (3 + 5) / (2 * 1024) = 2^-8
    g = [oracle.f32_to_fp16(np.array([3.0], np.float32)), oracle.f32_to_fp16(np.array([5.0], np.float32))]
    assert oracle.all_reduce_mean(g, FP16, 2.0 * 1024.0)[0] == np.float32(2.0 ** -8)


def test_negative_zero_sums_to_positive_zero():
    g = [_bf16([-0.0])] * 4
    out = oracle.all_reduce_mean(g, BF16, 4.0)
    assert out.view(np.uint32)[0] == 0


def test_all_gather_places_shards_at_their_offsets():
    psi, n_d, pad = 10, 3, 2
    S = oracle.shard_size(psi, n_d, pad)       # 4
    shards = [np.full(S, 100 + r, dtype=np.uint16) for r in range(n_d)]
    got = oracle.all_gather_u16(shards, psi, S)
    assert list(got) == [100] * 4 + [101] * 4 + [102] * 2
