"""The allocation-free fused step, for callers that cannot allocate device
memory: plug-ins inside a framework that owns all device memory, services
that forbid allocation once running (a cudaMalloc may synchronise the
device), programs whose memory is committed up front to a fixed pool.

zero_step_fused_noalloc replaces the caller's workspace with a scratch array
inside the library.  Through the C ABI, on two calls in a row, it must give
exactly the bits zero_step_fused gives with a caller-allocated workspace (the
kernels are the same and deterministic; only the workspace's address
differs), and the oracle's bits; it must leave the free device memory as it
was, and refuse a request its scratch cannot hold.  This file is collected
last on purpose: it must pass alone in a fresh process and after the rest of
the suite."""
import ctypes

import pytest
import torch

import zero_optimizer_step_02_gb300 as z
from gpu_helpers import Job

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().contiguous().view(torch.uint8)


@pytest.mark.parametrize("n_d,clip", [(8, 1.0), (4, 1.0), (8, 0.0)])
def test_noalloc_step_matches_the_workspace_step(n_d, clip):
    # n_d = 8 with clipping keeps the reduced gradient in the scratch; n_d = 4
    # re-reads the ranks and needs only the partial sums; no clipping needs none
    psi = 1_000_003
    hp = z.hparams(lr=3e-4, beta1=0.9, beta2=0.95, weight_decay=0.1, max_norm=clip)
    job = Job(psi, n_d, hp=hp, seed=5)                     # the no-alloc side, checked against the oracle
    assert job.plan.workspace_bytes(hp) <= z.NOALLOC_SCRATCH_BYTES
    ref = z.StepBuffers(job.plan, hp, device="cuda")       # zero_step_fused with a caller's workspace
    ref.master.copy_(job.buf.master)
    ref.init_scalars()
    nws = job.buf
    for step in (1, 2):                                    # two calls in a row
        job.new_grads(step, sigma=1e-2, heavy_tail=True)
        ref.grads.copy_(nws.grads)
        z.zero_step_fused(job.plan.handle, hp, ref.rank_list(), ref.master, ref.m, ref.v, ref.master, ref.m, ref.v,
                          ref.lp, ref.scalars, ref.ws)
        z.zero_step_fused_noalloc(job.plan.handle, hp, nws.rank_list(), nws.master, nws.m, nws.v, nws.master,
                                  nws.m, nws.v, nws.lp, nws.scalars)
        torch.cuda.synchronize()
        for a, b in ((nws.master, ref.master), (nws.m, ref.m), (nws.v, ref.v), (nws.lp, ref.lp)):
            assert torch.equal(_bits(a), _bits(b))
        s_ref, s_nws = ref.scalars_host(), nws.scalars_host()
        assert s_nws.t == s_ref.t == step and s_nws.status == 0
        assert s_nws.sqnorm == s_ref.sqnorm and s_nws.clip_coef == s_ref.clip_coef
        job.oracle_step()
        job.settle()


def test_noalloc_step_leaves_free_device_memory_unchanged():
    psi, n_d = 500_001, 8
    hp = z.hparams(lr=1e-3, max_norm=1.0)
    job = Job(psi, n_d, hp=hp, seed=9)
    b = job.buf
    job.new_grads(1, sigma=1e-2)

    def call():
        z.zero_step_fused_noalloc(job.plan.handle, hp, b.rank_list(), b.master, b.m, b.v, b.master, b.m, b.v, b.lp,
                                  b.scalars)

    call()                      # the first call looks up the scratch (and loads the kernels)
    torch.cuda.synchronize()
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0 and torch.cuda.memory_allocated() == alloc0
    assert b.scalars_host().t == 4


def test_noalloc_step_refuses_what_its_scratch_cannot_hold():
    # clipping with n_d > 4 keeps 4 * n_d * S bytes of reduced gradient: 2^21
    # parameters need 8 MB, more than the 4 MB the scratch holds
    psi, n_d = 1 << 21, 8
    hp = z.hparams(max_norm=1.0)
    plan = z.Plan(psi, n_d, stage=2, shard_pad=8)
    assert plan.workspace_bytes(hp) > z.NOALLOC_SCRATCH_BYTES
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
    # without clipping nothing of the scratch is needed: any size is accepted
    assert plan.workspace_bytes(z.hparams()) <= z.NOALLOC_SCRATCH_BYTES
