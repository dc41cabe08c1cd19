"""CPU pins of the check the GPU tests make when a clipped step's clip
coefficient comes out one fp32 ulp away from the oracle's (the GPU sums the
squared norm in another order): they re-run the oracle's Adam from the state
before the step on the oracle's reduced gradient times the GPU's coefficient
(tests/gpu_helpers.py: step_with_coef, accum_ghat, Job.ghat) and compare bit
for bit.  That re-run must be the oracle's own step whenever it is given the
oracle's own coefficient -- for the plain, the quantized-exchange and the
accumulated step -- and a coefficient one ulp away must change the result
(else the check would accept anything)."""
import types

import numpy as np
import pytest

import oracle
from gpu_helpers import accum_ghat, step_with_coef


def _rows(n_d, psi, seed, sigma=1e-2):
    rng = np.random.default_rng(seed)
    return [oracle.f32_to_lp((rng.standard_normal(psi) * sigma).astype(np.float32), oracle.BF16)
            for _ in range(n_d)]


def _state(n_d, psi, pad, seed):
    S = oracle.shard_size(psi, n_d, pad)
    rng = np.random.default_rng(seed)
    master = np.zeros(n_d * S, np.float32)
    master[:psi] = (rng.standard_normal(psi) * 0.02).astype(np.float32)
    return oracle.State(master, np.zeros(n_d * S, np.float32), np.zeros(n_d * S, np.float32),
                        oracle.new_scalars(1.0)), S


def _next_ulp(x, d):
    return (np.float32(x).view(np.int32) + np.int32(d)).view(np.float32)


def _same(st, master, m, v):
    return all(np.array_equal(a.view(np.uint32), b.view(np.uint32)) for a, b in
               ((st.master, master), (st.m, m), (st.v, v)))


@pytest.mark.parametrize("n_d,psi,pad", [(2, 30_001, 8), (8, 50_003, 1), (5, 4097, 64)])
def test_rerun_with_the_oracle_coefficient_is_the_oracle_step(n_d, psi, pad):
    hp = oracle.hparams(lr=3e-4, beta2=0.95, weight_decay=0.1, max_norm=0.05)
    st, S = _state(n_d, psi, pad, seed=psi)
    for step in range(1, 4):
        rows = _rows(n_d, psi, seed=100 * step + n_d)
        pre = st.copy()
        gathered = np.zeros(psi, np.uint16)
        assert not oracle.zero_step(rows, oracle.BF16, hp, st, pad, 2, gathered=gathered)
        coef = np.float32(st.scalars.clip_coef)
        assert coef < 1.0
        g_hat = oracle.reduce_scatter(rows, oracle.BF16, float(n_d), S)
        got, lp = step_with_coef(pre, g_hat, coef, hp, st.scalars.beta1_pow, st.scalars.beta2_pow, psi, oracle.BF16)
        assert _same(got, st.master, st.m, st.v) and np.array_equal(lp, gathered)
        # one ulp either way gives another result (the comparison has teeth)
        for d in (-1, 1):
            other, _ = step_with_coef(pre, g_hat, _next_ulp(coef, d), hp, st.scalars.beta1_pow,
                                      st.scalars.beta2_pow, psi, oracle.BF16)
            assert not np.array_equal(other.m.view(np.uint32), st.m.view(np.uint32))


def test_rerun_matches_the_quantized_exchange_step():
    n_d, psi, pad = 8, 40_001, 16
    hp = oracle.hparams(lr=3e-4, beta2=0.95, weight_decay=0.1, max_norm=0.5)
    st, S = _state(n_d, psi, pad, seed=3)
    for step in range(1, 3):
        rows = _rows(n_d, psi, seed=7 + step)
        codes, scales = oracle.quantize_ranks(rows, psi, S, 2048)
        pre = st.copy()
        gathered = np.zeros(psi, np.uint16)
        assert not oracle.zero_step_qgz(codes, scales, 2048, hp, st, pad, 2, psi, gathered=gathered)
        coef = np.float32(st.scalars.clip_coef)
        assert coef < 1.0
        g_hat = oracle.reduce_scatter_q(codes, scales, psi, S, 2048, float(n_d))
        got, lp = step_with_coef(pre, g_hat, coef, hp, st.scalars.beta1_pow, st.scalars.beta2_pow, psi, oracle.BF16)
        assert _same(got, st.master, st.m, st.v) and np.array_equal(lp, gathered)


@pytest.mark.parametrize("loss_scaling", [False, True])
def test_rerun_matches_the_accumulated_step(loss_scaling):
    n_d, psi, pad, k = 4, 20_011, 8, 3
    hp = oracle.hparams(lr=1e-3, max_norm=0.05, loss_scaling=loss_scaling)
    st, S = _state(n_d, psi, pad, seed=11)
    scale = 1024.0 if loss_scaling else 1.0
    st.scalars = oracle.new_scalars(scale)
    acc = None
    for mu in range(1, k):
        acc = oracle.accumulate_grads(_rows(n_d, psi, seed=mu, sigma=1e-2 * scale), oracle.BF16, acc)
    rows = _rows(n_d, psi, seed=k, sigma=1e-2 * scale)
    pre = st.copy()
    gathered = np.zeros(psi, np.uint16)
    assert not oracle.zero_step_accum(rows, oracle.BF16, acc, k, hp, st, pad, 2, gathered=gathered)
    coef = np.float32(st.scalars.clip_coef)
    assert coef < 1.0
    job = types.SimpleNamespace(rows=rows, gdt=0, n_d=n_d, pre=pre,
                                hp=types.SimpleNamespace(loss_scaling=int(loss_scaling)))
    g_hat = accum_ghat(job, acc, k)
    got, lp = step_with_coef(pre, g_hat, coef, hp, st.scalars.beta1_pow, st.scalars.beta2_pow, psi, oracle.BF16)
    assert _same(got, st.master, st.m, st.v) and np.array_equal(lp, gathered)
