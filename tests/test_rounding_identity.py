"""The block quantizer's kernels round with an addition instead of rintf:
t = fl(y + 1.5 * 2^23), r = fl(t - 1.5 * 2^23), the code byte is t's low
byte, and y is near a tie when |fl(y - r)| >= 0.5 - 2^-14.  These CPU tests
check, in IEEE float32 (numpy), that this gives the round-half-even integer
and the same tie decisions as the floor-based form, exhaustively over every
mantissa of the exponents the codes use and on random floats of any size."""
import numpy as np
import pytest

M = np.float32(12582912.0)          # 1.5 * 2^23
BAND = np.float32(0.49993896484375)  # 0.5 - 2^-14
HALF_BAND = np.float32(6.103515625e-05)


def _check(y):
    y = y.astype(np.float32)
    t = (y + M).astype(np.float32)
    r = (t - M).astype(np.float32)
    small = np.abs(y) < np.float32(4194304.0)     # |y| < 2^22
    # rint with ties to even
    assert np.array_equal(r[small], np.rint(y[small]))
    # the low byte of t is the two's-complement low byte of rint(y)
    code = np.rint(y[small]).astype(np.int64)
    assert np.array_equal(t[small].view(np.uint32) & 0xFF, (code & 0xFF).astype(np.uint32))
    # the tie test agrees with |(y - floor(y)) - 1/2| <= 2^-14 wherever that one is exact
    near_new = ~(np.abs((y - r).astype(np.float32)) < BAND)
    f = (y - np.floor(y)).astype(np.float32)
    exact = (f.astype(np.float64) == (y.astype(np.float64) - np.floor(y.astype(np.float64))))
    near_old = np.abs((f - np.float32(0.5)).astype(np.float32)) <= HALF_BAND
    sel = small & exact
    assert np.array_equal(near_new[sel], near_old[sel])
    # large magnitudes stay beyond +-127.5, so the clamp maps them as it maps rint(y)
    big = ~small & np.isfinite(y)
    assert np.all(np.sign(r[big]) == np.sign(y[big])) and np.all(np.abs(r[big]) > 127.5)


@pytest.mark.parametrize("e", range(-2, 8))
def test_every_mantissa_of_the_code_range(e):
    # all 2^23 floats of [2^e, 2^(e+1)), both signs: |y| from 0.25 to 256
    m = np.arange(1 << 23, dtype=np.uint32)
    bits = ((np.uint32(127 + e) << 23) | m).astype(np.uint32)
    y = bits.view(np.float32)
    _check(y)
    _check(-y)


def test_random_floats_of_any_size():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 32, size=4_000_000, dtype=np.uint64).astype(np.uint32)
    y = bits.view(np.float32)
    _check(y[np.isfinite(y)])


def test_small_values_and_zero():
    y = np.concatenate([np.array([0.0, -0.0, 0.5, -0.5, 1.5, 2.5, -2.5, 127.5, -127.5], np.float32),
                        np.linspace(-0.25, 0.25, 100_001, dtype=np.float32)])
    _check(y)
