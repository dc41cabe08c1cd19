"""C-ABI tests that need no GPU: the library builds and loads, exports every
function include/zero.h declares, and its host logic (plans, accounting,
argument checks) behaves.  No call here reaches a kernel launch: every call
that takes device pointers is made to fail its argument checks first."""
import ctypes
import os
import re

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def z():
    import __graft_entry__
    __graft_entry__.build()
    import zero_optimizer_step_02_gb300 as z
    return z


def _declared():
    with open(os.path.join(ROOT, "include", "zero.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"ZERO_API\s+[\w\s\*]+?\b(zero_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(z):
    names = _declared()
    assert len(names) >= 18
    lib = z._capi.library()
    for n in names:
        assert hasattr(lib, n), n
    # and the binding offers each under the same name
    for n in names:
        assert hasattr(z._capi, n), n


def test_abi_and_struct_layout(z):
    assert z.zero_abi_version() == 2
    assert z.zero_dev_scalars_size() == ctypes.sizeof(z.ZeroDevScalars) == 64
    assert z.zero_status_str(0) == "ok"
    assert "misaligned" in z.zero_status_str(2)


@pytest.mark.parametrize("psi,n_d,pad", [(1, 1, 1), (1_000_003, 4, 8), (1_000_003, 4, 1), (7, 8, 8),
                                         (124_439_808, 8, 8), (268_435_456, 64, 8), (218_112_000, 16, 8),
                                         (5, 3, 4096)])
def test_plan_layout_matches_the_oracle(z, psi, n_d, pad):
    p = z.Plan(psi, n_d, stage=2, shard_pad=pad)
    S = oracle.shard_size(psi, n_d, pad)
    assert p.shard == S and p.padded == n_d * S
    assert p.valid_len == [oracle.valid_len(psi, S, r) for r in range(n_d)]


@pytest.mark.parametrize("stage", [0, 1, 2, 3])
@pytest.mark.parametrize("psi,n_d", [(7.5e9, 64), (1.3e9, 8), (1.5e9, 1), (124_439_808, 8)])
def test_plan_accounting_matches_the_oracle(z, stage, psi, n_d):
    p = z.Plan(int(psi), n_d, stage=2)
    got = p.memory(stage)
    want = oracle.model_state_bytes(int(psi), n_d, stage)
    assert got == pytest.approx(want, rel=1e-15)
    assert p.comm_volume(stage) == oracle.comm_volume(stage) * int(psi)


def test_stage_table_from_the_library(z):
    # "ZeRO (딥 러닝)", ZeRO-DP의 세 단계: 120 / 31.4 / 16.6 / 1.9 GB at 7.5B, 64 GPUs
    p = z.Plan(7_500_000_000, 64, stage=2)
    assert [round(p.memory(s)[3] / 1e9, 1) for s in range(4)] == [120.0, 31.4, 16.6, 1.9]


def test_workspace_size(z):
    hp = z.hparams()
    p = z.Plan(1000, 8, stage=2)
    base = p.workspace_bytes(hp)
    assert base >= 8 * 4096 and base % 256 == 0
    assert p.workspace_bytes(z.hparams(max_norm=1.0)) == base + 4 * p.padded   # n_d > 4: reduced grad in ws
    p4 = z.Plan(1000, 4, stage=2)
    assert p4.workspace_bytes(z.hparams(max_norm=1.0)) == base                  # n_d <= 4: re-read instead


@pytest.mark.parametrize("args", [(0, 4, 2, 0, 8), (10, 0, 2, 0, 8), (10, 257, 2, 0, 8), (10, 4, 0, 0, 8),
                                  (10, 4, 4, 0, 8), (10, 4, 2, 2, 8), (10, 4, 2, 0, 0), (10, 4, 2, 0, 4097)])
def test_plan_rejects_bad_arguments(z, args):
    with pytest.raises(z.ZeroError) as e:
        z.zero_plan_create(*args)
    assert e.value.status == 1


def test_bucket_rounding_and_param_dtype(z):
    p = z.Plan(10_000_000, 8, stage=2, param_dtype=z.ZERO_FP16, reduce_bucket_elems=1000)
    assert p.param_dtype == z.ZERO_FP16
    with pytest.raises(z.ZeroError):
        z.zero_plan_create_ex(100, 2, 2, 0, 8, param_dtype=7)


def _raw(z, name, *args):
    return z._capi.raw_status(name, *args)


def test_calls_check_arguments_before_touching_the_device(z):
    hp = z.hparams()
    p = z.Plan(1000, 2, stage=2)
    h = p.handle
    A = 0x10000          # 16- and 256-byte aligned fake addresses: never dereferenced,
    B = 0x20000          # every call below fails its checks first
    S1, S2, S3 = 0x100000, 0x200000, 0x300000   # distinct state arrays
    ranks_ok = (ctypes.c_void_p * 2)(A, B)
    ranks_bad = (ctypes.c_void_p * 2)(A, B + 2)
    ranks_null = (ctypes.c_void_p * 2)(A, None)
    hpp = ctypes.byref(hp)
    # NULL plan / hparams
    assert _raw(z, "zero_step_fused", None, hpp, ranks_ok, A, A, A, A, A, A, A, A, A, None) == 1
    assert _raw(z, "zero_step_fused", h, None, ranks_ok, A, A, A, A, A, A, A, A, A, None) == 1
    # misaligned rank pointer, NULL rank pointer
    assert _raw(z, "zero_step_fused", h, hpp, ranks_bad, A, A, A, A, A, A, A, A, A, None) == 2
    assert _raw(z, "zero_step_fused", h, hpp, ranks_null, A, A, A, A, A, A, A, A, A, None) == 1
    # misaligned state, partly aliased state
    assert _raw(z, "zero_step_fused", h, hpp, ranks_ok, A + 4, A, A, A, A, A, A, A, A, None) == 2
    assert _raw(z, "zero_step_fused", h, hpp, ranks_ok, A, A, A, A, B, B, A, A, A, None) == 1
    # scalars not 256-aligned
    assert _raw(z, "zero_step_fused", h, hpp, ranks_ok, A, A, A, A, A, A, A, A + 16, A, None) == 2
    # bad hyper-parameters
    bad = z.hparams(beta1=1.0)
    assert _raw(z, "zero_step_fused", h, ctypes.byref(bad), ranks_ok, A, A, A, A, A, A, A, A, A, None) == 1
    nan = z.hparams(lr=float("nan"))
    assert _raw(z, "zero_adam_shard_step", h, ctypes.byref(nan), A, A, A, A, A, A, None) == 1
    ls = z.hparams(loss_scaling=True, scale_window=0)
    assert _raw(z, "zero_reduce_scatter", h, ranks_ok, ctypes.byref(ls), A, A, A, None) == 1
    # workspace required with clipping
    clip = z.hparams(max_norm=1.0)
    assert _raw(z, "zero_step_fused", h, ctypes.byref(clip), ranks_ok, S1, S2, S3, S1, S2, S3, A, A, None,
                None) == 1
    # quantized gather: block limits, fused variant only with block 2048 and no clipping
    assert _raw(z, "zero_quant_gather", h, A, 31, A, A, A, None) == 1
    assert _raw(z, "zero_quant_gather", h, A, 70000, A, A, A, None) == 1
    assert _raw(z, "zero_step_fused_qgather", h, hpp, ranks_ok, A, A, A, A, A, A, 1024, A, A, A, A, A, None) == 3
    # clipping or loss scaling need the workspace; loss scaling needs the state in place
    assert _raw(z, "zero_step_fused_qgather", h, ctypes.byref(clip), ranks_ok, S1, S2, S3, S1, S2, S3, 2048, A, A, A,
                A, None, None) == 1
    lsc = z.hparams(loss_scaling=True)
    assert _raw(z, "zero_step_fused_qgather", h, ctypes.byref(lsc), ranks_ok, S1, S2, S3, B, B + 0x4000, B + 0x8000,
                2048, A, A, A,
                A, A, None) == 3
    # the timeout probe rejects limits outside (0, 10 s]
    assert _raw(z, "zero_debug_wait_timeout", A, 0, None) == 1
    assert _raw(z, "zero_debug_wait_timeout", A, 20_000_000_000, None) == 1
    assert _raw(z, "zero_debug_stream_timeout", 0, A + 8, A, 1000, None) == 2
    assert _raw(z, "zero_debug_stream_timeout", 0, A, A + 16, 1000, None) == 2
    assert _raw(z, "zero_debug_stream_timeout", 0, A, A, 0, None) == 1
    assert _raw(z, "zero_debug_stream_timeout", 4, A, A, 1000, None) == 1
    # fp16 parameters cannot take the bf16 quantizer
    p16 = z.Plan(1000, 2, stage=2, param_dtype=z.ZERO_FP16)
    assert _raw(z, "zero_quant_gather", p16.handle, A, 2048, A, A, A, None) == 3


def test_library_is_built_in_tree(z):
    assert os.path.dirname(z._capi.LIB_PATH) == os.path.join(ROOT, "zero_optimizer_step_02_gb300")


def test_quantized_gradient_exchange_argument_checks(z):
    A = 0x10000
    S1, S2, S3 = 0x100000, 0x200000, 0x300000   # distinct state arrays (updated in place)
    p = z.Plan(1000, 2, stage=2)
    ranks = (ctypes.c_void_p * 2)(A, A)
    hp = z.hparams()
    clip = z.hparams(max_norm=1.0)
    assert _raw(z, "zero_quantize_grads", p.handle, ranks, 31, ranks, A, None, None) == 1
    assert _raw(z, "zero_quantize_grads", p.handle, ranks, 2048, (ctypes.c_void_p * 2)(A, A + 8), A, None, None) == 2
    assert _raw(z, "zero_quantize_grads", p.handle, ranks, 2048, ranks, A, A + 16, None) == 2
    p16 = z.Plan(1000, 2, stage=2, grad_dtype=z.ZERO_FP16)
    assert _raw(z, "zero_quantize_grads", p16.handle, ranks, 2048, ranks, A, None, None) == 3
    assert _raw(z, "zero_step_fused_qgz", p.handle, ctypes.byref(hp), ranks, A, 1024, S1, S2, S3, S1, S2, S3, A, A,
                None, None) == 3
    # clipping needs the workspace; bf16 gradients take no loss scaling
    assert _raw(z, "zero_step_fused_qgz", p.handle, ctypes.byref(clip), ranks, A, 2048, S1, S2, S3, S1, S2, S3, A, A,
                None, None) == 1
    assert _raw(z, "zero_step_fused_qgz", p.handle, ctypes.byref(clip), ranks, A, 2048, S1, S2, S3, S1, S2, S3, A, A,
                A + 16, None) == 2
    lsc = z.hparams(loss_scaling=True)
    assert _raw(z, "zero_step_fused_qgz", p.handle, ctypes.byref(lsc), ranks, A, 2048, S1, S2, S3, S1, S2, S3, A, A,
                A, None) == 3


def test_gradient_accumulation_argument_checks(z):
    A, B = 0x10000, 0x20000
    p = z.Plan(1000, 2, stage=2)
    ranks = (ctypes.c_void_p * 2)(A, B)
    hp = z.hparams()
    hpp = ctypes.byref(hp)
    # accumulate: misaligned out / in, partly overlapping in and out, misaligned scalars
    assert _raw(z, "zero_accumulate_grads", p.handle, ranks, None, A + 4, None, None) == 2
    assert _raw(z, "zero_accumulate_grads", p.handle, ranks, A + 8, B, None, None) == 2
    assert _raw(z, "zero_accumulate_grads", p.handle, ranks, A, A + 16, None, None) == 1
    assert _raw(z, "zero_accumulate_grads", p.handle, ranks, A, B, A + 16, None) == 2
    assert _raw(z, "zero_accumulate_grads", None, ranks, A, B, None, None) == 1
    # the accumulated step: micro-batch count in [1, 65536], acc given exactly when k > 1
    for acc, k in ((A, 1), (None, 2), (A, 0), (A, 65537)):
        assert _raw(z, "zero_step_fused_accum", p.handle, hpp, ranks, acc, k, A, A, A, A, A, A, A, A, A, None) == 1
    assert _raw(z, "zero_step_fused_accum", p.handle, hpp, ranks, A + 4, 2, A, A, A, A, A, A, A, A, A, None) == 2


def test_prebuilt_rank_pointer_arrays(z):
    # a pointer array built once by rank_ptrs goes through unchanged and
    # reaches the same argument checks as a list of addresses
    hp = z.hparams()
    plan = z.Plan(1000, 2, stage=2)     # kept alive: its handle is freed with it
    h = plan.handle
    A, B = 0x10000, 0x20000
    arr = z.rank_ptrs([A, B + 2])
    assert list(arr) == [A, B + 2]
    assert z._capi._ptr_array(arr) is arr
    for ranks in (arr, [A, B + 2]):
        with pytest.raises(z.ZeroError) as e:
            z.zero_step_fused(h, hp, ranks, A, A, A, A, A, A, A, A, A, stream=0)
        assert e.value.status == 2


def test_two_exchange_step_argument_checks(z):
    # every case fails its checks before anything is launched
    A = 0x10000
    S1, S2, S3 = 0x100000, 0x200000, 0x300000   # distinct state arrays (updated in place)
    p = z.Plan(1000, 2, stage=2)
    ranks = (ctypes.c_void_p * 2)(A, A)
    f = "zero_step_fused_qgz_qgather"
    hp, clip, lsc = z.hparams(), z.hparams(max_norm=1.0), z.hparams(loss_scaling=True)
    assert _raw(z, f, p.handle, ctypes.byref(hp), ranks, A, 1024, S1, S2, S3, S1, S2, S3, A, A, A, A, None, None) == 3
    assert _raw(z, f, p.handle, ctypes.byref(lsc), ranks, A, 2048, S1, S2, S3, S1, S2, S3, A, A, A, A, A, None) == 3
    assert _raw(z, f, p.handle, ctypes.byref(clip), ranks, A, 2048, S1, S2, S3, S1, S2, S3, A, A, A, A, None, None) == 1
    assert _raw(z, f, p.handle, ctypes.byref(hp), ranks, A, 2048, S1, S2, S3, S1, S2, S3, A + 4, A, A, A, None, None) == 2
    assert _raw(z, f, p.handle, ctypes.byref(hp), ranks, A, 2048, S1, S2, S3, S1, S2, S3, A, A, A, A + 16, None,
                None) == 2
    p16 = z.Plan(1000, 2, stage=2, param_dtype=z.ZERO_FP16)
    assert _raw(z, f, p16.handle, ctypes.byref(hp), ranks, A, 2048, S1, S2, S3, S1, S2, S3, A, A, A, A, None, None) == 3


def test_overlapping_state_arrays_are_refused(z):
    # master/m/v (n_d*S floats each) may be updated in place, array by array;
    # any other shared byte between an output and another state array is refused
    hp = z.hparams()
    plan = z.Plan(1000, 2, stage=2)          # n_d*S = 1008 floats = 4032 bytes
    h, hpp = plan.handle, ctypes.byref(hp)
    A = 0x10000
    ranks = (ctypes.c_void_p * 2)(A, A)
    S1, S2, S3 = 0x100000, 0x200000, 0x300000
    T1, T2, T3 = 0x400000, 0x500000, 0x600000

    def step(*state):
        return _raw(z, "zero_step_fused", h, hpp, ranks, *state, A, A, A, None)
    assert step(S1, S2, S3, S1, S2, S3 + 4096) == 1           # partly in place
    assert step(S1, S2, S3, T1, T1 + 1024, T3) == 1            # two outputs share bytes
    assert step(S1, S2, S3, T1, T2, S1 + 2048) == 1            # an output overlaps another input
    assert step(S1, S1 + 2048, S3, S1, S1 + 2048, S3) == 1     # in place, but m overlaps master
    assert _raw(z, "zero_adam_shard_step", h, hpp, A, S1, S1 + 16, S3, None, A, None) == 1   # m overlaps master


def test_noalloc_scratch_size_matches_the_header(z):
    # the binding's constant is the header's ZERO_NOALLOC_SCRATCH_BYTES
    with open(os.path.join(ROOT, "include", "zero.h")) as f:
        m = re.search(r"#define ZERO_NOALLOC_SCRATCH_BYTES \((\d+)u \+ (\d+)u \* \(1u << (\d+)\)\)", f.read())
    assert m is not None
    a, b, c = (int(x) for x in m.groups())
    assert z.NOALLOC_SCRATCH_BYTES == a + b * (1 << c)


def test_layer_loop_argument_checks(z):
    A, B = 0x10000, 0x20000
    S1, S2, S3, LP, ACC = 0x100000, 0x200000, 0x300000, 0x400000, 0x500000
    hp = z.hparams(lr=1e-3)
    p3 = z.Plan(1000, 2, stage=3)
    p3b = z.Plan(2000, 2, stage=3)
    p2 = z.Plan(1000, 2, stage=2)
    p4 = z.Plan(1000, 4, stage=3)
    ranks = (ctypes.c_void_p * 2)(A, B)
    ranks4 = (ctypes.c_void_p * 4)(A, B, A, B)
    gathered = (ctypes.c_void_p * 2)(A, B)

    def stack(*plans, acc=None):
        arr = (z.ZeroLayer * len(plans))()
        for i, p in enumerate(plans):
            r = ranks4 if p is p4 else ranks
            arr[i] = z.ZeroLayer(p.handle, ctypes.cast(r, ctypes.c_void_p), acc, S1, S2, S3, LP, None, None, 0)
        return arr

    def call(h, layers, gathers=1, n_gathered=2, g=gathered, sc=A, ws=None, k=1, codes=None, scales=None):
        return _raw(z, "zero_step_layers", ctypes.byref(h), len(layers), layers, k, gathers, n_gathered, g, codes,
                    scales, sc, ws, None, None)

    # clipping or loss scaling need the workspace (256-byte aligned)
    clip, ls = z.hparams(max_norm=1.0), z.hparams(loss_scaling=True)
    assert call(clip, stack(p3, p3b)) == 1
    assert call(ls, stack(p3, p3b)) == 1
    assert call(clip, stack(p3, p3b), ws=A + 16) == 2
    # only stage-3 plans, all with the same n_d
    assert call(hp, stack(p3, p2)) == 1
    assert call(hp, stack(p3, p4)) == 1
    # gathers 1 or 2; 1 <= n_gathered <= n_layers; aligned buffers and scalars
    assert call(hp, stack(p3, p3b), gathers=3) == 1
    assert call(hp, stack(p3, p3b), n_gathered=0) == 1
    assert call(hp, stack(p3, p3b), n_gathered=3) == 1
    assert call(hp, stack(p3, p3b), g=(ctypes.c_void_p * 2)(A, B + 8)) == 2
    assert call(hp, stack(p3, p3b), sc=A + 16) == 2
    # a misaligned shard buffer
    bad = stack(p3, p3b)
    bad[1].shards_lp = LP + 2
    assert call(hp, bad) == 2
    # accumulation: acc given exactly when micro_batches > 1, 16-byte aligned
    assert call(hp, stack(p3, p3b), k=2) == 1
    assert call(hp, stack(p3, p3b, acc=ACC), k=1) == 1
    assert call(hp, stack(p3, p3b, acc=ACC + 4), k=2) == 2
    assert call(hp, stack(p3, p3b), k=0) == 1
    # quantized gathers: codes and scales for every buffer, or none; bf16 parameters only
    arr2 = (ctypes.c_void_p * 2)(A, B)
    assert call(hp, stack(p3, p3b), codes=arr2) == 1
    assert call(hp, stack(p3, p3b), scales=arr2) == 1
    assert call(hp, stack(p3, p3b), codes=arr2, scales=(ctypes.c_void_p * 2)(A, B + 4)) == 2
    p16a, p16b = z.Plan(1000, 2, stage=3, param_dtype=z.ZERO_FP16), z.Plan(2000, 2, stage=3, param_dtype=z.ZERO_FP16)
    assert call(hp, stack(p16a, p16b), codes=arr2, scales=arr2) == 3
    # state in host memory must be page-locked host memory (these addresses are not)
    host = stack(p3, p3b)
    host[0].state_on_host = 1
    assert call(hp, host) == 1
    host[0].state_on_host = 2
    assert call(hp, host) == 1


def test_layer_loop_workspace_size(z):
    # per layer room for its reduce pass's partial sums; with clipping and
    # n_d > 4 each layer's fp32 reduced gradient too (256-byte aligned)
    p8a, p8b = z.Plan(10_000, 8, stage=3), z.Plan(3_001, 8, stage=3)
    p2 = z.Plan(10_000, 2, stage=3)
    layers8 = [(p8a.handle, [0x10000] * 8, 0x100000, 0x200000, 0x300000, 0x400000),
               (p8b.handle, [0x10000] * 8, 0x100000, 0x200000, 0x300000, 0x400000)]
    part = 2 * 32768
    assert z.zero_layers_workspace_bytes(z.hparams(), layers8) == part
    assert z.zero_layers_workspace_bytes(z.hparams(loss_scaling=True), layers8) == part
    want = part + sum((4 * p.padded + 255) // 256 * 256 for p in (p8a, p8b))
    assert z.zero_layers_workspace_bytes(z.hparams(max_norm=1.0), layers8) == want
    layers2 = [(p2.handle, [0x10000] * 2, 0x100000, 0x200000, 0x300000, 0x400000)]
    assert z.zero_layers_workspace_bytes(z.hparams(max_norm=1.0), layers2) == 32768
