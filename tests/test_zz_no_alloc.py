"""The allocation-free fused step, for callers that cannot allocate device
memory (code that runs where cudaMalloc is not allowed, such as inside a CUDA
graph capture without a memory pool; programs whose device memory belongs to
another allocator; services that forbid allocation once running).

zero_step_fused_noalloc replaces the caller's workspace with a scratch array
inside the library.  Through the C ABI it must give what zero_step_fused
gives with a caller-allocated workspace, on two calls in a row, within the
tolerance the parity tests use (relative 1e-6 on master/m/v, 1 ulp on the
16-bit parameters), and refuse a request its scratch cannot hold.  This file
is collected last on purpose: it must pass alone in a fresh process and
after the rest of the suite."""
import ctypes

import numpy as np
import pytest
import torch

import zero_optimizer_step_02_gb300 as z
from gpu_helpers import u16
from zero_optimizer_step_02_gb300 import synth

pytestmark = pytest.mark.gpu


def _within_tolerance(a, b, rel=1e-6):
    a64, b64 = a.astype(np.float64), b.astype(np.float64)
    denom = max(float(np.max(np.abs(b64))), 1e-30)
    return float(np.max(np.abs(a64 - b64))) / denom <= rel


def _lp_within_one_ulp(x, y):
    same = (x >> 15) == (y >> 15)
    d = np.abs(x.astype(np.int64) - y.astype(np.int64))
    return bool(np.all(d[same] <= 1) and np.all((x[~same] & 0x7FFF) + (y[~same] & 0x7FFF) <= 1))


@pytest.mark.parametrize("n_d,clip", [(8, 1.0), (4, 1.0), (8, 0.0)])
def test_noalloc_step_matches_the_workspace_step(n_d, clip):
    # n_d = 8 with clipping keeps the reduced gradient in the scratch; n_d = 4
    # re-reads the ranks and needs only the partial sums; no clipping needs none
    psi = 1_000_003
    hp = z.hparams(lr=3e-4, beta1=0.9, beta2=0.95, weight_decay=0.1, max_norm=clip)
    plan = z.Plan(psi, n_d, stage=2, shard_pad=8)
    assert plan.workspace_bytes(hp) <= 32768 + 4 * (1 << 20)
    ref = z.StepBuffers(plan, hp, device="cuda")            # caller-allocated workspace
    nws = z.StepBuffers(plan, hp, device="cuda")            # its workspace is never passed
    master = synth.master_init(plan.padded, psi, seed=5, device="cuda")
    for b in (ref, nws):
        b.master.copy_(master)
        b.init_scalars()
    for step in (1, 2):                                     # two calls in a row
        g = synth.rank_grads(n_d, psi, 1e-2, seed=17, step=step, device="cuda", heavy_tail=True,
                             row_pad=ref.grads.shape[1] - psi)
        ref.grads.copy_(g)
        nws.grads.copy_(g)
        z.zero_step_fused(plan.handle, hp, ref.rank_list(), ref.master, ref.m, ref.v, ref.master, ref.m, ref.v,
                          ref.lp, ref.scalars, ref.ws)
        z.zero_step_fused_noalloc(plan.handle, hp, nws.rank_list(), nws.master, nws.m, nws.v, nws.master, nws.m,
                                  nws.v, nws.lp, nws.scalars)
        torch.cuda.synchronize()
        for a, b in ((nws.master, ref.master), (nws.m, ref.m), (nws.v, ref.v)):
            assert _within_tolerance(a.cpu().numpy(), b.cpu().numpy())
        assert _lp_within_one_ulp(u16(nws.lp[:psi]), u16(ref.lp[:psi]))
        s_ref, s_nws = ref.scalars_host(), nws.scalars_host()
        assert s_nws.t == s_ref.t == step and s_nws.status == 0
        assert s_nws.sqnorm == pytest.approx(s_ref.sqnorm, rel=1e-12)


def test_noalloc_step_refuses_what_its_scratch_cannot_hold():
    # clipping with n_d > 4 keeps 4 * n_d * S bytes of reduced gradient: 2^21
    # parameters need 8 MB, more than the 4 MB the scratch holds
    psi, n_d = 1 << 21, 8
    hp = z.hparams(max_norm=1.0)
    plan = z.Plan(psi, n_d, stage=2, shard_pad=8)
    A = 0x10000   # never dereferenced: the size check comes before anything else
    ranks = (ctypes.c_void_p * n_d)(*([A] * n_d))
    st = z._capi.raw_status("zero_step_fused_noalloc", plan.handle, ctypes.byref(hp), ranks, A, A, A, A, A, A,
                            A, A, None)
    assert st == 6   # ZERO_ERR_BOUNDS
    with pytest.raises(z.ZeroError) as e:
        buf = z.StepBuffers(z.Plan(4096, n_d, stage=2), hp, device="cuda")
        z.zero_step_fused_noalloc(plan.handle, hp, [buf.grads[0]] * n_d, buf.master, buf.m, buf.v, buf.master,
                                  buf.m, buf.v, buf.lp, buf.scalars)
    assert e.value.status == 6
