"""An independent NumPy float32 restatement of the update the oracle
computes, compared with the oracle bit for bit.

The pages print no Adam equations.  The reading (textbook Adam, Kingma & Ba,
evaluated in the efficient order of their Section 2, with decoupled weight
decay as in AdamW) fixes every fp32 operation and its order:

    per step:   b1^t, b2^t    fp64 running products of the fp32 betas
                bc1 = fp32(1 - b1^t), bc2 = fp32(1 - b2^t), s = sqrt(bc2)
                step = (lr * s) / bc1,  eps_hat = eps * s
                omb1 = 1 - b1, omb2 = 1 - b2, decay = 1 - lr * wd
    per element p = p * decay                  (only when wd != 0)
                m = b1 * m + omb1 * g
                v = b2 * v + omb2 * (g * g)
                p = p - step * (m / (sqrt(v) + eps_hat))

each binary operation one IEEE float32 rounding.  NumPy float32 scalars and
arrays round every operation that way and never fuse a multiply into an add,
so the code below is the reading written out again, sharing nothing with the
oracle's C.  The 50-digit comparison with Algorithm 1 pins the mathematics;
this pins the operation order: a reordering the decimal test tolerates
(eps added before the division by s, the step size formed as lr / bc1 * s,
the product m * (1 / denom)) changes bits here.

The reduction in front of it is restated too: the mean of the ranks' bf16
gradients, summed in fp32 in rank order from +0 and divided once by N_d."""
import numpy as np
import pytest

import oracle

F = np.float32


def _consts(lr, b1, b2, eps, wd, b1p, b2p):
    bc1 = F(1.0 - b1p)
    bc2 = F(1.0 - b2p)
    s = np.sqrt(bc2)
    step = (F(lr) * s) / bc1
    eps_hat = F(eps) * s
    return step, eps_hat, F(1) - F(b1), F(1) - F(b2), F(1) - F(lr) * F(wd)


def _adam_f32(lr, b1, b2, eps, wd, b1p, b2p, g, p, m, v):
    step, eps_hat, omb1, omb2, decay = _consts(lr, b1, b2, eps, wd, b1p, b2p)
    g = g.astype(F)
    if F(wd) != 0:
        p = p * decay
    m = F(b1) * m + omb1 * g
    v = F(b2) * v + omb2 * (g * g)
    p = p - step * (m / (np.sqrt(v) + eps_hat))
    return p, m, v


def _bits(a):
    return np.asarray(a, dtype=F).view(np.uint32)


HPARAMS = [dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0),
           dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1),
           dict(lr=1e-2, beta1=0.5, beta2=0.75, eps=1e-6, weight_decay=0.01),
           dict(lr=0.1, beta1=0.0, beta2=0.0, eps=1e-3, weight_decay=0.5)]


@pytest.mark.parametrize("hpd", HPARAMS)
@pytest.mark.parametrize("seed", range(5))
def test_adam_matches_a_float32_restatement_bit_for_bit(hpd, seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 9))                  # Psi <= 8
    hp = oracle.hparams(**hpd)
    p0 = rng.normal(0, 0.02, n).astype(F)
    p, m, v = p0.copy(), np.zeros(n, F), np.zeros(n, F)
    q, mq, vq = p0.copy(), np.zeros(n, F), np.zeros(n, F)
    b1p = b2p = 1.0
    for _ in range(6):
        # gradients over several magnitudes, with zeros and signs mixed in
        g = (rng.normal(0, 1, n) * 10.0 ** rng.integers(-6, 1, n)).astype(F)
        g[rng.random(n) < 0.15] = 0
        b1p *= float(F(hpd["beta1"]))
        b2p *= float(F(hpd["beta2"]))
        oracle.adam_update(hp, oracle.adam_consts(hp, b1p, b2p), g, p, m, v)
        q, mq, vq = _adam_f32(hpd["lr"], hpd["beta1"], hpd["beta2"], hpd["eps"], hpd["weight_decay"], b1p, b2p, g,
                              q, mq, vq)
        assert np.array_equal(_bits(p), _bits(q)) and np.array_equal(_bits(m), _bits(mq))
        assert np.array_equal(_bits(v), _bits(vq))


def _mean_bf16(rows, n_d):
    acc = np.zeros(rows[0].size, F)               # +0.0, then ranks in order
    for r in rows:
        acc = acc + (r.astype(np.uint32) << 16).view(F)
    return acc / F(n_d)


@pytest.mark.parametrize("n_d", [1, 2, 3, 8])
def test_plain_step_matches_the_restatement(n_d):
    # the whole plain data-parallel step of the oracle (all-reduce mean ->
    # Adam -> bf16 cast) over several steps against the restatement
    rng = np.random.default_rng(100 + n_d)
    psi = 7
    hpd = HPARAMS[1]
    hp = oracle.hparams(**hpd)
    st = oracle.State(rng.normal(0, 0.02, psi).astype(F), np.zeros(psi, F), np.zeros(psi, F), oracle.new_scalars())
    q, mq, vq = st.master.copy(), np.zeros(psi, F), np.zeros(psi, F)
    b1p = b2p = 1.0
    for _ in range(4):
        rows = [oracle.f32_to_bf16(rng.normal(0, 1e-2, psi).astype(F)) for _ in range(n_d)]
        skipped, lp = oracle.plain_dp_step(rows, oracle.BF16, hp, st)
        assert not skipped
        b1p *= float(F(hpd["beta1"]))
        b2p *= float(F(hpd["beta2"]))
        q, mq, vq = _adam_f32(hpd["lr"], hpd["beta1"], hpd["beta2"], hpd["eps"], hpd["weight_decay"], b1p, b2p,
                              _mean_bf16(rows, n_d), q, mq, vq)
        assert np.array_equal(_bits(st.master), _bits(q)) and np.array_equal(_bits(st.m), _bits(mq))
        assert np.array_equal(_bits(st.v), _bits(vq))
        # bf16 round-to-nearest-even of the updated master, by torch's cast
        import torch
        want = torch.from_numpy(q).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(lp, want)
