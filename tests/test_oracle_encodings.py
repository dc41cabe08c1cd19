"""Pins of the oracle's 16-bit encodings against library routines (numpy's
IEEE half conversion, torch's bfloat16 cast), exhaustively where the domain is
small and on a seeded sample of fp32 bit patterns otherwise."""
import numpy as np
import pytest
import torch

import oracle


def _sample_f32_bits(n, seed):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    edge = np.array([0x00000000, 0x80000000, 0x7F800000, 0xFF800000, 0x00000001, 0x807FFFFF,
                     0x3F800000, 0x3F808000, 0x3F818000, 0x3F807FFF, 0x3F808001, 0x7F7FFFFF,
                     0x7F7F8000, 0x477FE000, 0x477FEFFF, 0x477FF000, 0x477FF001, 0x38800000,
                     0x387FFFFF, 0x33800000, 0x33800001, 0x33000000, 0x33000001, 0x337FFFFF,
                     0x38000000, 0x38001000], dtype=np.uint32)
    return np.concatenate([edge, bits])


def _not_nan(bits):
    return (bits & 0x7FFFFFFF) <= 0x7F800000


@pytest.mark.parametrize("seed", [1, 2])
def test_bf16_matches_torch(seed):
    bits = _sample_f32_bits(400_000, seed)
    bits = bits[_not_nan(bits)]
    x = bits.view(np.float32)
    want = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.f32_to_bf16(x)
    assert np.array_equal(got, want)


def test_bf16_exhaustive_round_trip():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = oracle.bf16_to_f32(h)
    want = torch.from_numpy(h.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(f), nan)
    assert np.array_equal(f[~nan].view(np.uint32), want[~nan].view(np.uint32))
    assert np.array_equal(oracle.f32_to_bf16(f[~nan]), h[~nan])


@pytest.mark.parametrize("seed", [3, 4])
def test_fp16_matches_numpy(seed):
    bits = _sample_f32_bits(400_000, seed)
    bits = bits[_not_nan(bits)]
    # concentrate half of the sample in and around fp16's range, subnormals included
    rng = np.random.default_rng(seed + 100)
    near = rng.uniform(-30, 17, size=200_000)
    sign = rng.choice([-1.0, 1.0], size=near.size)
    x = np.concatenate([bits.view(np.float32), (sign * 2.0 ** near).astype(np.float32)])
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.f32_to_fp16(x), want)


def test_fp16_exhaustive_decode():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = oracle.fp16_to_f32(h)
    want = h.view(np.float16).astype(np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(f), nan)
    assert np.array_equal(f[~nan].view(np.uint32), want[~nan].view(np.uint32))
    assert np.array_equal(oracle.f32_to_fp16(f[~nan]), h[~nan])


def test_nan_stays_nan():
    x = np.array([np.nan, -np.nan], dtype=np.float32)
    assert np.all(np.isnan(oracle.bf16_to_f32(oracle.f32_to_bf16(x))))
    assert np.all(np.isnan(oracle.fp16_to_f32(oracle.f32_to_fp16(x))))
