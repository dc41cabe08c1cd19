"""Seeded synthetic inputs for the ZeRO-DP step (rank gradients, initial
master weights, injected non-finite values).

This module draws random numbers and casts them to the requested dtype with
torch; it holds none of the method's arithmetic.  The tests hand the very same
bytes to the CUDA path and to the CPU oracle.  Recipe: each (seed, step, rank)
gets its own torch generator; gradients are N(0, sigma) (sigma the standard
deviation), optionally with a heavy tail (each element independently, with
probability 0.01, multiplied by 100 before the cast) and optionally multiplied
by a loss scale before the cast to fp16; master weights are N(0, 0.02) fp32.
"""
import torch

_CHUNK = 1 << 26  # elements generated at a time (bounds the fp32 temporary)


def _gen(device, *key):
    g = torch.Generator(device=device)
    h = 1469598103934665603
    for k in key:
        h = ((h ^ (int(k) & 0xFFFFFFFFFFFF)) * 1099511628211) & 0x7FFFFFFFFFFFFFFF
    g.manual_seed(h)
    return g


def gaussian_(out, sigma, seed, *key, heavy_tail=False, scale=1.0):
    """Fill the 1-D tensor `out` (bf16 / fp16 / fp32) in place with seeded draws."""
    n = out.numel()
    dev = out.device
    g = _gen(dev, seed, *key)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        x = torch.randn(hi - lo, generator=g, device=dev, dtype=torch.float32) * sigma
        if heavy_tail:
            tail = torch.rand(hi - lo, generator=g, device=dev) < 0.01
            x = torch.where(tail, x * 100.0, x)
        if scale != 1.0:
            x = x * scale
        out[lo:hi].copy_(x)
    return out


def rank_grads(n_d, psi, sigma, seed, step, dtype=torch.bfloat16, device="cpu", heavy_tail=False, scale=1.0,
               row_pad=0):
    """A [n_d, psi + row_pad] tensor; row r is rank r's gradient (first psi used)."""
    buf = torch.zeros(n_d, psi + row_pad, dtype=dtype, device=device)
    for r in range(n_d):
        gaussian_(buf[r, :psi], sigma, seed, step, r, heavy_tail=heavy_tail, scale=scale)
    return buf


def master_init(n, psi, seed, sigma=0.02, device="cpu"):
    """fp32 master weights of n entries: N(0, sigma) in [0, psi), +0 padding."""
    m = torch.zeros(n, dtype=torch.float32, device=device)
    gaussian_(m[:psi], sigma, seed, 0xFFFF)
    return m


def pick_index(seed, step, n_d, psi):
    """A seeded (rank, index) for an injected non-finite value."""
    g = _gen("cpu", seed, step, 0xBAD)
    r = int(torch.randint(0, n_d, (1,), generator=g))
    j = int(torch.randint(0, psi, (1,), generator=g))
    return r, j
