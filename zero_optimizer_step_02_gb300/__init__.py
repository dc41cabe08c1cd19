"""GB300-native ZeRO-DP optimizer step.

The compute lives in libzero.so (hand-written CUDA for sm_103a behind a C
ABI, declared in include/zero.h).  This package is the thin Python side:

* ``_capi``   -- one function per C entry point, same names, marshalling only;
* ``Plan``    -- owns a plan handle and its layout numbers;
* ``StepBuffers`` -- allocates the device buffers of one simulated job with
  torch (rank gradients, fp32 master/m/v, 16-bit parameters, workspace,
  step scalars) -- allocation only, no arithmetic;
* ``synth``   -- seeded synthetic inputs.

Importing this package fails if libzero.so has not been built.
"""
import ctypes

from . import _capi
from ._capi import (NOALLOC_SCRATCH_BYTES, ZERO_BF16, ZERO_FP16, ZERO_DEV_TIMEOUT, ZeroDevScalars, ZeroError, ZeroHparams, hparams,
                    zero_abi_version, zero_adam_shard_step, zero_all_gather, zero_debug_wait_timeout,
                    zero_dev_scalars_size, zero_grad_sqnorm, zero_launch_count, zero_plan_comm_volume, zero_plan_create,
                    zero_plan_create_ex, zero_plan_destroy, zero_plan_memory, zero_plan_query, zero_quant_gather,
                    zero_reduce_scatter, zero_scalars_init, zero_status_str, zero_step_fused,
                    zero_step_fused_noalloc, zero_step_fused_qgather, zero_workspace_bytes,
                    zero_quantize_grads, zero_step_fused_qgz, zero_step_fused_offload, zero_accumulate_grads,
                    zero_step_fused_accum, zero_debug_stream_timeout, zero_step_fused_qgz_qgather, rank_ptrs,
                    zero_step_layers, zero_layers_workspace_bytes, LayerStack, ZeroLayer)

__all__ = ["Plan", "StepBuffers", "read_scalars", "row_len", "hparams", "rank_ptrs", "ZeroError", "ZeroHparams",
           "LayerStack", "ZeroLayer",
           "ZERO_BF16", "ZERO_FP16", "ZERO_DEV_TIMEOUT", "NOALLOC_SCRATCH_BYTES"] + [n for n in dir(_capi) if n.startswith("zero_")]


class Plan:
    """A plan handle (host memory) plus its layout: S, n_d*S, valid lengths."""

    def __init__(self, psi, n_d, stage=2, grad_dtype=ZERO_BF16, shard_pad=8, param_dtype=None,
                 reduce_bucket_elems=0):
        self.handle = zero_plan_create_ex(psi, n_d, stage, grad_dtype, shard_pad, param_dtype,
                                          reduce_bucket_elems)
        self.psi, self.n_d, self.stage = psi, n_d, stage
        self.grad_dtype = grad_dtype
        self.param_dtype = ZERO_BF16 if param_dtype is None else param_dtype
        self.shard_pad = shard_pad
        self.shard, self.padded, self.valid_len = zero_plan_query(self.handle, n_d)

    def memory(self, stage=None, k=12.0):
        return zero_plan_memory(self.handle, self.stage if stage is None else stage, k)

    def comm_volume(self, stage=None):
        return zero_plan_comm_volume(self.handle, self.stage if stage is None else stage)

    def workspace_bytes(self, hp):
        return zero_workspace_bytes(self.handle, hp)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value:
            zero_plan_destroy(h)
            self.handle = None


def row_len(psi, extra=0):
    """Elements per rank row of a [n_d, row] gradient tensor: psi rounded up
    to 8 (16-byte aligned rows) plus `extra`."""
    return (psi + 7) // 8 * 8 + extra


def _torch_dtype(dt):
    import torch
    return torch.bfloat16 if dt == ZERO_BF16 else torch.float16


class StepBuffers:
    """Device buffers of one simulated data-parallel job, allocated with torch.

    grads    [n_d, row] 16-bit rank gradients (row >= psi, 16-byte aligned rows)
    master, m, v   fp32 [n_d*S]   (a second set when pingpong=True)
    lp       16-bit parameters: gathered [psi] (stages 1-2) or sharded [n_d*S] (stage 3)
    ws       workspace bytes, scalars 64 bytes (256-aligned torch allocations)
    """

    def __init__(self, plan, hp, device="cuda", pingpong=False, row_extra=0, grads=None):
        import torch
        self.plan = plan
        n = plan.padded
        if grads is None:
            grads = torch.zeros(plan.n_d, row_len(plan.psi, row_extra), dtype=_torch_dtype(plan.grad_dtype),
                                device=device)
        self.grads = grads
        self.master = torch.zeros(n, dtype=torch.float32, device=device)
        self.m = torch.zeros(n, dtype=torch.float32, device=device)
        self.v = torch.zeros(n, dtype=torch.float32, device=device)
        self.pingpong = pingpong
        if pingpong:
            self.master2 = torch.zeros_like(self.master)
            self.m2 = torch.zeros_like(self.m)
            self.v2 = torch.zeros_like(self.v)
        lp_n = n if plan.stage == 3 else plan.psi
        self.lp = torch.zeros(max(lp_n, 8), dtype=_torch_dtype(plan.param_dtype), device=device)
        self.ws = torch.zeros(max(plan.workspace_bytes(hp), 256), dtype=torch.uint8, device=device)
        self.scalars = torch.zeros(256, dtype=torch.uint8, device=device)

    def rank_list(self):
        return [self.grads[r] for r in range(self.plan.n_d)]

    def rank_ptrs(self):
        """The ranks' rows as the pointer array the entry points read, built
        once per grads tensor (again if grads is replaced)."""
        key = (self.grads.data_ptr(), self.grads.stride(0))
        if getattr(self, "_rank_key", None) != key:
            self._rank_arr, self._rank_key = rank_ptrs(self.rank_list()), key
        return self._rank_arr

    def init_scalars(self, loss_scale=1.0):
        zero_scalars_init(self.scalars, loss_scale)

    def step(self, hp, stream=None):
        """One fused step; with pingpong the state alternates between the two sets."""
        if self.pingpong:
            zero_step_fused(self.plan.handle, hp, self.rank_ptrs(), self.master, self.m, self.v, self.master2,
                            self.m2, self.v2, self.lp, self.scalars, self.ws, stream)
            self.master, self.master2 = self.master2, self.master
            self.m, self.m2 = self.m2, self.m
            self.v, self.v2 = self.v2, self.v
        else:
            zero_step_fused(self.plan.handle, hp, self.rank_ptrs(), self.master, self.m, self.v, self.master,
                            self.m, self.v, self.lp, self.scalars, self.ws, stream)

    def accumulate(self, first, stream=None):
        """Add the micro-batch now in grads to the fp32 accumulator `acc`
        (padded length; started from +0 when first)."""
        import torch
        if getattr(self, "acc", None) is None:
            self.acc = torch.zeros(self.plan.padded, dtype=torch.float32, device=self.master.device)
        zero_accumulate_grads(self.plan.handle, self.rank_ptrs(), None if first else self.acc, self.acc,
                              self.scalars, stream)

    def step_accum(self, hp, micro_batches, stream=None):
        """The step at the last of micro_batches micro-batches (grads holds
        it; acc the sum of the earlier ones)."""
        acc = None if micro_batches == 1 else self.acc
        zero_step_fused_accum(self.plan.handle, hp, self.rank_ptrs(), acc, micro_batches, self.master, self.m,
                              self.v, self.master, self.m, self.v, self.lp, self.scalars, self.ws, stream)

    def scalars_host(self):
        return read_scalars(self.scalars)


def read_scalars(scalars_tensor):
    """Copy the 64-byte device scalars block to the host (synchronising) and
    return it as a ZeroDevScalars."""
    raw = bytes(scalars_tensor[:ctypes.sizeof(ZeroDevScalars)].cpu().numpy().tobytes())
    return ZeroDevScalars.from_buffer_copy(raw)
