"""Pins of the oracle's Adam against the mathematics.

The pages print no Adam equations; the reading is textbook Adam (Kingma & Ba,
Algorithm 1: bias-corrected moments, eps outside the square root) with
decoupled weight decay (Loshchilov & Hutter, AdamW).  The oracle evaluates it
in fp32 with a fixed operation order; these tests check it against

* the textbook update evaluated in 50-digit decimal arithmetic on tiny inputs
  (the exact result up to the fp32 rounding the oracle is allowed), and
* closed forms and special cases: step one from a zero state, a constant
  gradient, lr = 0, a zero gradient, beta = 0, decay alone, and eps when
  |g| is comparable to it.

A dropped bias correction, eps inside the root, a wrong sign or a coupled
decay each fail at least one of them."""
import decimal
from decimal import Decimal

import numpy as np
import pytest

import oracle

decimal.getcontext().prec = 50


def _f32(x):
    return float(np.float32(x))


def _textbook(hp, p0, g_steps, wd):
    """Textbook AdamW in 50-digit decimals from the same fp32 inputs."""
    lr, b1, b2, eps = (Decimal(_f32(v)) for v in (hp.lr, hp.beta1, hp.beta2, hp.eps))
    wd = Decimal(_f32(wd))
    p = [Decimal(float(x)) for x in p0]
    m = [Decimal(0)] * len(p)
    v = [Decimal(0)] * len(p)
    for t, g in enumerate(g_steps, start=1):
        for i, gi in enumerate(g):
            gi = Decimal(float(gi))
            m[i] = b1 * m[i] + (1 - b1) * gi
            v[i] = b2 * v[i] + (1 - b2) * gi * gi
            mhat = m[i] / (1 - b1 ** t)
            vhat = v[i] / (1 - b2 ** t)
            p[i] = p[i] - lr * wd * p[i] - lr * mhat / (vhat.sqrt() + eps)
    return [float(x) for x in p], [float(x) for x in m], [float(x) for x in v]


def _run_oracle(hp, p0, g_steps):
    p = np.array(p0, dtype=np.float32)
    m = np.zeros_like(p)
    v = np.zeros_like(p)
    b1p = b2p = 1.0
    for g in g_steps:
        b1p *= float(np.float32(hp.beta1))
        b2p *= float(np.float32(hp.beta2))
        c = oracle.adam_consts(hp, b1p, b2p)
        oracle.adam_update(hp, c, np.asarray(g, np.float32), p, m, v)
    return p, m, v


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("wd", [0.0, 0.1])
@pytest.mark.parametrize("betas", [(0.9, 0.999), (0.9, 0.95), (0.5, 0.75)])
def test_against_textbook_adam_in_decimals(seed, wd, betas):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 9))
    steps = int(rng.integers(1, 6))
    hp = oracle.hparams(lr=float(rng.choice([1e-3, 3e-4, 1e-2])), beta1=betas[0], beta2=betas[1],
                        eps=1e-8, weight_decay=wd)
    p0 = rng.normal(0, 0.02, n).astype(np.float32)
    gs = [rng.normal(0, float(rng.choice([1e-3, 1e-1, 3.0])), n).astype(np.float32) for _ in range(steps)]
    p, m, v = _run_oracle(hp, p0, gs)
    tp, tm, tv = _textbook(hp, p0, gs, wd)
    # m, v: a handful of fp32 roundings per step
    assert np.allclose(m, tm, rtol=2e-6 * steps, atol=0)
    assert np.allclose(v, tv, rtol=2e-6 * steps, atol=0)
    # p: the change p - p0 is what Adam computes; allow a few ulp of p plus a
    # relative error on the change
    dp_true = np.array(tp) - p0.astype(np.float64)
    err = np.abs(p.astype(np.float64) - np.array(tp))
    ulp = np.spacing(np.abs(p)).astype(np.float64)
    assert np.all(err <= 2 * steps * ulp + 1e-5 * np.abs(dp_true)), (err, ulp, dp_true)


@pytest.mark.parametrize("g", [3e-3, -2.5e-1, 7.0, -1e-5])
def test_step_one_from_zero_state_is_lr_times_sign(g):
    # m1 = (1-b1) g, v1 = (1-b2) g^2  =>  mhat = g, vhat = g^2, update = lr g / (|g| + eps)
    hp = oracle.hparams(lr=1e-3)
    p, m, v = _run_oracle(hp, [0.25], [[g]])
    want = 0.25 - _f32(1e-3) * g / (abs(g) + _f32(1e-8))
    assert p[0] == pytest.approx(want, rel=0, abs=4 * np.spacing(np.float32(0.25)))
    assert m[0] == pytest.approx((1 - _f32(0.9)) * g, rel=1e-6)
    assert v[0] == pytest.approx((1 - _f32(0.999)) * g * g, rel=1e-6)


def test_constant_gradient_moves_lr_per_step():
    # with a constant g the bias-corrected moments are exactly g and g^2 at every step
    hp = oracle.hparams(lr=1e-3, beta1=0.9, beta2=0.999)
    g, T = 0.05, 25
    p, _, _ = _run_oracle(hp, [1.0], [[g]] * T)
    want = 1.0 - T * _f32(1e-3) * g / (g + _f32(1e-8))
    assert p[0] == pytest.approx(want, abs=T * 4 * np.spacing(np.float32(1.0)))


def test_lr_zero_keeps_master_and_updates_moments():
    hp = oracle.hparams(lr=0.0)
    p0 = np.array([0.5, -0.25, 3.0], np.float32)
    g = np.array([1e-3, -2.0, 0.0], np.float32)
    p, m, v = _run_oracle(hp, p0, [g])
    assert np.array_equal(p.view(np.uint32), p0.view(np.uint32))
    assert np.array_equal(m, np.float32(1 - np.float32(0.9)) * g)
    assert np.array_equal(v, np.float32(1 - np.float32(0.999)) * (g * g))


def test_zero_gradient_is_a_no_op():
    hp = oracle.hparams(lr=1e-2)
    p0 = np.array([0.5, -0.25, 0.0, 1e-30], np.float32)
    p, m, v = _run_oracle(hp, p0, [np.zeros(4, np.float32)] * 3)
    assert np.array_equal(p.view(np.uint32), p0.view(np.uint32))
    assert not m.any() and not v.any()


def test_zero_betas_make_every_step_a_first_step():
    hp = oracle.hparams(lr=1e-2, beta1=0.0, beta2=0.0)
    gs = [[0.3], [-2.0], [1e-4]]
    p, _, _ = _run_oracle(hp, [0.0], gs)
    want = -sum(_f32(1e-2) * g[0] / (abs(g[0]) + _f32(1e-8)) for g in gs)
    assert p[0] == pytest.approx(want, abs=1e-8)


def test_decay_alone_is_repeated_multiplication():
    hp = oracle.hparams(lr=3e-4, weight_decay=0.1)
    p0 = np.array([0.7, -1.3], np.float32)
    p, _, _ = _run_oracle(hp, p0, [np.zeros(2, np.float32)] * 10)
    decay = np.float32(1) - np.float32(np.float32(3e-4) * np.float32(0.1))
    want = p0.copy()
    for _ in range(10):
        want = (want * decay).astype(np.float32)
    assert np.array_equal(p, want)


def test_eps_is_outside_the_square_root():
    # |g| = eps: update = lr * g / (|g| + eps) = lr / 2.  With eps under the root
    # it would be lr * g / sqrt(g^2 + eps) ~ lr * 1e-4, far off.
    hp = oracle.hparams(lr=1e-3, eps=1e-8)
    g = _f32(1e-8)
    p, _, _ = _run_oracle(hp, [0.0], [[g]])
    assert p[0] == pytest.approx(-_f32(1e-3) * g / (g + _f32(1e-8)), rel=1e-5)
    assert p[0] == pytest.approx(-5e-4, rel=1e-5)


def test_gradient_sign_moves_against_the_gradient():
    hp = oracle.hparams(lr=1e-3)
    p, _, _ = _run_oracle(hp, [0.0, 0.0], [[2.0, -2.0]])
    assert p[0] < 0 < p[1]
