"""Pins of the oracle's quantized gradient exchange (ZeRO++ qgZ reading):
lossless on the int8 grid it must reproduce the plain ZeRO step bit for bit;
its codes are the pinned block quantizer's; the reconstructed average stays
within half a quantization step per rank of the exact one."""
import numpy as np
import pytest

import oracle
from oracle import BF16


def _on_grid_grads(n_d, psi, S, block, e, seed):
    """bf16 gradients k * 2^-e with |k| <= 127 and one |k| = 127 in every
    block of every shard, so the block scale is exactly 2^-e."""
    rng = np.random.default_rng(seed)
    rows = []
    for _ in range(n_d):
        k = rng.integers(-127, 128, size=psi).astype(np.float64)
        for r in range(n_d):
            L = oracle.valid_len(psi, S, r)
            for lo in range(0, L, block):
                k[r * S + lo] = 127 * rng.choice([-1, 1])
        rows.append(oracle.f32_to_bf16((k * 2.0 ** -e).astype(np.float32)))
    return rows


@pytest.mark.parametrize("n_d,psi,pad,block", [(2, 5000, 8, 2048), (4, 1003, 1, 256), (8, 7000, 64, 2048),
                                               (3, 4096 * 3 + 5, 8, 2048)])
@pytest.mark.parametrize("stage", [2, 3])
@pytest.mark.parametrize("max_norm", [0.0, 0.05])      # plain, and clipped (active on these inputs)
def test_lossless_on_grid_equals_the_plain_step(n_d, psi, pad, block, stage, max_norm):
    S = oracle.shard_size(psi, n_d, pad)
    hp = oracle.hparams(lr=1e-3, weight_decay=0.01, max_norm=max_norm)
    a = oracle.State(np.zeros(n_d * S, np.float32), np.zeros(n_d * S, np.float32),
                     np.zeros(n_d * S, np.float32), oracle.new_scalars())
    a.master[:psi] = np.random.default_rng(1).normal(0, 0.02, psi).astype(np.float32)
    b = a.copy()
    for step in range(3):
        rows = _on_grid_grads(n_d, psi, S, block, 10 + step, seed=step)
        codes, scales = oracle.quantize_ranks(rows, psi, S, block)
        used = scales[:, :n_d][scales[:, :n_d] != 0]
        assert np.all(used == np.float32(2.0 ** -(10 + step)))
        assert not scales[:, n_d:].any()          # rank padding of the layout
        bufs_a = dict(lp_shards=np.zeros(n_d * S, np.uint16), gathered=np.zeros(psi, np.uint16))
        bufs_b = dict(lp_shards=np.zeros(n_d * S, np.uint16), gathered=np.zeros(psi, np.uint16))
        oracle.zero_step(rows, BF16, hp, a, pad, stage, **bufs_a)
        oracle.zero_step_qgz(codes, scales, block, hp, b, pad, stage, psi, **bufs_b)
        for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v)):
            assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
        if max_norm > 0:
            assert a.scalars.clip_coef < 1.0 and a.scalars.clip_coef == b.scalars.clip_coef
        key = "lp_shards" if stage == 3 else "gathered"
        assert np.array_equal(bufs_a[key], bufs_b[key])


@pytest.mark.parametrize("n_d,psi,pad,block", [(2, 10_000, 8, 2048), (5, 3001, 1, 512)])
def test_codes_are_the_block_quantizers(n_d, psi, pad, block):
    S = oracle.shard_size(psi, n_d, pad)
    rng = np.random.default_rng(psi)
    rows = [oracle.f32_to_bf16(rng.normal(0, 1e-3, psi).astype(np.float32)) for _ in range(n_d)]
    codes, scales = oracle.quantize_ranks(rows, psi, S, block)
    for q in range(n_d):
        flat = np.zeros(n_d * S, np.uint16)
        flat[:psi] = rows[q]
        c, s, _ = oracle.quant_gather(flat, n_d, psi, S, block)
        assert np.array_equal(codes[q][:psi], c[:psi])
        assert np.array_equal(scales[:, q], s)


@pytest.mark.parametrize("n_d", [1, 2, 8])
def test_reconstruction_error_is_within_half_a_step_per_rank(n_d):
    psi, pad, block = 20_000, 8, 2048
    S = oracle.shard_size(psi, n_d, pad)
    rng = np.random.default_rng(n_d)
    rows = [oracle.f32_to_bf16(rng.normal(0, 1e-3, psi).astype(np.float32)) for _ in range(n_d)]
    codes, scales = oracle.quantize_ranks(rows, psi, S, block)
    got = oracle.reduce_scatter_q(codes, scales, psi, S, block, float(n_d))
    exact = np.mean([oracle.bf16_to_f32(r).astype(np.float64) for r in rows], axis=0)
    nbs = -(-S // block)
    j = np.arange(psi)
    sidx = (j // S) * nbs + (j % S) // block
    half = np.sum(scales[sidx, :n_d].astype(np.float64), axis=1) / 2.0 / n_d
    err = np.abs(got[:psi].astype(np.float64) - exact)
    # half a step per rank, plus the fp32 roundings of n_d products, n_d sums and one division
    assert np.all(err <= half * (1 + 1e-6) + (2 * n_d + 2) * 2.0 ** -24 * np.abs(exact) + 1e-30)
    if n_d == 1:
        # one rank: the average is exactly the dequantized value code * scale
        want = np.array([np.float32(codes[0][i]) * scales[sidx[i], 0] for i in range(psi)], np.float32)
        assert np.array_equal(got[:psi], want)


def test_rank_order_decides_the_rounding():
    # one shard-block holds elements 0 and 1 (psi = 6, n_d = 3, S = 2).
    # rank 0: 127 * 2^-6 (sets s = 2^-6) and 64 * 2^-6 = 1; ranks 1, 2:
    # 127 * 2^-30 and 64 * 2^-30 = 2^-24.  Dequantized and added in rank order:
    # (1 + 2^-24) ties to 1, again 1 -> fl(1/3); in reverse 1 + 2^-23.
    psi, n_d, pad, block = 6, 3, 2, 2048
    S = oracle.shard_size(psi, n_d, pad)
    assert S == 2
    vals = [[127 * 2.0 ** -6, 1.0], [127 * 2.0 ** -30, 2.0 ** -24], [127 * 2.0 ** -30, 2.0 ** -24]]
    rows = []
    for v in vals:
        x = np.zeros(psi, np.float32)
        x[:2] = v
        rows.append(oracle.f32_to_bf16(x))
    codes, scales = oracle.quantize_ranks(rows, psi, S, block)
    assert [int(c[1]) for c in codes] == [64, 64, 64]
    got = oracle.reduce_scatter_q(codes, scales, psi, S, block, 3.0)
    assert got[1] == np.float32(1.0) / np.float32(3.0)
    rev = oracle.reduce_scatter_q(codes[::-1], np.ascontiguousarray(scales[:, [2, 1, 0, 3]]), psi, S, block, 3.0)
    assert rev[1] == np.float32(1.0 + 2.0 ** -23) / np.float32(3.0)


def test_point_reduction_matches_the_shard_reduction():
    # the sampled-point form used by the full-size checks computes the same
    # values as the reduce-scatter form at every point
    psi, n_d, pad, block = 9000, 4, 8, 2048
    S = oracle.shard_size(psi, n_d, pad)
    rng = np.random.default_rng(2)
    rows = [oracle.f32_to_bf16(rng.normal(0, 1e-3, psi).astype(np.float32)) for _ in range(n_d)]
    codes, scales = oracle.quantize_ranks(rows, psi, S, block)
    full = oracle.reduce_scatter_q(codes, scales, psi, S, block, float(n_d))
    nbs = -(-S // block)
    j = np.arange(psi)
    row = (j // S) * nbs + (j % S) // block
    pts = oracle.reduce_points_q([c[:psi] for c in codes], [scales[row, q] for q in range(n_d)], float(n_d))
    assert np.array_equal(pts.view(np.uint32), full[:psi].view(np.uint32))
