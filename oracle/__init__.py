"""CPU oracle of the ZeRO-DP optimizer step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never calls it and
shares no code with it.

This module marshals numpy arrays into the plain single-threaded C oracle
(``zero_oracle.c``).  16-bit floats travel as their raw ``uint16`` bit patterns.
Every function names, in its C source, the page and section it follows.
"""
import ctypes
import os
from dataclasses import dataclass, field

import numpy as np

from . import build as _build

BF16 = 0
FP16 = 1

_u16p = ctypes.POINTER(ctypes.c_uint16)
_f32p = ctypes.POINTER(ctypes.c_float)
_i8p = ctypes.POINTER(ctypes.c_int8)


class Hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("max_norm", ctypes.c_float), ("loss_scaling", ctypes.c_int),
                ("scale_window", ctypes.c_int), ("min_scale", ctypes.c_float)]


class Scalars(ctypes.Structure):
    _fields_ = [("t", ctypes.c_longlong), ("beta1_pow", ctypes.c_double),
                ("beta2_pow", ctypes.c_double), ("loss_scale", ctypes.c_float),
                ("good_steps", ctypes.c_int), ("overflow", ctypes.c_int),
                ("sqnorm", ctypes.c_double), ("clip_coef", ctypes.c_float)]


class AdamConsts(ctypes.Structure):
    _fields_ = [("step_size", ctypes.c_float), ("eps_hat", ctypes.c_float), ("omb1", ctypes.c_float),
                ("omb2", ctypes.c_float), ("decay", ctypes.c_float)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        # ZERO_ORACLE_LIB points at another build of the oracle (the mutation
        # test uses it to check that the pins catch planted mistakes)
        path = os.environ.get("ZERO_ORACLE_LIB") or _build.build()
        L = ctypes.CDLL(path)
        ll, i32, f32, f64, vp = (ctypes.c_longlong, ctypes.c_int, ctypes.c_float,
                                 ctypes.c_double, ctypes.c_void_p)
        sig = {
            "zo_shard_size": (ll, [ll, i32, i32]),
            "zo_valid_len": (ll, [ll, ll, i32]),
            "zo_owner": (None, [ll, ll, ctypes.POINTER(i32), ctypes.POINTER(ll)]),
            "zo_f32_to_bf16": (ctypes.c_uint16, [f32]),
            "zo_bf16_to_f32": (f32, [ctypes.c_uint16]),
            "zo_f32_to_fp16": (ctypes.c_uint16, [f32]),
            "zo_fp16_to_f32": (f32, [ctypes.c_uint16]),
            "zo_f32_to_lp_array": (None, [ll, _f32p, _u16p, i32]),
            "zo_lp_to_f32_array": (None, [ll, _u16p, _f32p, i32]),
            "zo_model_state_bytes": (None, [f64, f64, i32, f64, ctypes.POINTER(f64)]),
            "zo_comm_volume": (f64, [i32]),
            "zo_all_reduce_mean": (None, [i32, ll, vp, i32, f32, _f32p]),
            "zo_reduce_scatter": (None, [i32, ll, ll, vp, i32, f32, _f32p]),
            "zo_all_gather_u16": (None, [i32, ll, ll, vp, _u16p]),
            "zo_all_gather_f32": (None, [i32, ll, ll, vp, _f32p]),
            "zo_adam_consts_for": (None, [ctypes.POINTER(Hparams), f64, f64,
                                          ctypes.POINTER(AdamConsts)]),
            "zo_adam_update": (None, [ctypes.POINTER(Hparams), ctypes.POINTER(AdamConsts), ll,
                                      _f32p, _f32p, _f32p, _f32p]),
            "zo_sqnorm": (f64, [ll, _f32p]),
            "zo_clip_coef": (f32, [f32, f64, ctypes.POINTER(i32)]),
            "zo_plain_dp_step": (i32, [i32, ll, vp, i32, ctypes.POINTER(Hparams),
                                       ctypes.POINTER(Scalars), _f32p, _f32p, _f32p, _u16p, i32]),
            "zo_zero_step": (i32, [i32, ll, i32, i32, vp, i32, ctypes.POINTER(Hparams),
                                   ctypes.POINTER(Scalars), _f32p, _f32p, _f32p, _u16p, _u16p,
                                   i32]),
            "zo_scalars_init": (None, [ctypes.POINTER(Scalars), f32]),
            "zo_accumulate_grads": (None, [i32, ll, vp, i32, _f32p, _f32p]),
            "zo_zero_step_accum": (i32, [i32, ll, i32, i32, vp, i32, _f32p, i32, ctypes.POINTER(Hparams),
                                         ctypes.POINTER(Scalars), _f32p, _f32p, _f32p, _u16p, _u16p, i32]),
            "zo_quantize_block": (None, [ll, _u16p, _i8p, _f32p, _u16p]),
            "zo_quant_gather": (None, [i32, ll, ll, i32, _u16p, _i8p, _f32p, _u16p]),
            "zo_qgz_rank_stride": (ll, [i32]),
            "zo_reduce_points_q": (None, [i32, ll, vp, vp, f32, _f32p]),
            "zo_quantize_ranks": (None, [i32, ll, ll, i32, vp, vp, _f32p]),
            "zo_reduce_scatter_q": (None, [i32, ll, ll, i32, vp, _f32p, f32, _f32p]),
            "zo_zero_step_qgz": (i32, [i32, ll, i32, i32, i32, vp, _f32p, ctypes.POINTER(Hparams),
                                       ctypes.POINTER(Scalars), _f32p, _f32p, _f32p, _u16p, _u16p, i32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


# ---------------------------------------------------------------- helpers --
def _ptr(a, ctype):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _ptr_array(rows):
    """A C array of row pointers (keeps the numpy rows alive via the caller)."""
    arr = (ctypes.c_void_p * len(rows))()
    for i, r in enumerate(rows):
        assert r.flags["C_CONTIGUOUS"]
        arr[i] = r.ctypes.data
    return arr


def hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, max_norm=0.0,
            loss_scaling=False, scale_window=1000, min_scale=1.0):
    return Hparams(lr, beta1, beta2, eps, weight_decay, max_norm, int(bool(loss_scaling)),
                   scale_window, min_scale)


def new_scalars(loss_scale=1.0):
    sc = Scalars()
    lib().zo_scalars_init(ctypes.byref(sc), loss_scale)
    return sc


# ---------------------------------------------------------------- layout --
def shard_size(psi, n_d, shard_pad):
    return lib().zo_shard_size(psi, n_d, shard_pad)


def valid_len(psi, shard, r):
    return lib().zo_valid_len(psi, shard, r)


def owner(j, shard):
    r = ctypes.c_int()
    i = ctypes.c_longlong()
    lib().zo_owner(j, shard, ctypes.byref(r), ctypes.byref(i))
    return r.value, i.value


# ------------------------------------------------------------- encodings --
def f32_to_lp(x, dtype):
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    out = np.empty(x.size, dtype=np.uint16)
    lib().zo_f32_to_lp_array(x.size, _ptr(x, ctypes.c_float), _ptr(out, ctypes.c_uint16), dtype)
    return out


def lp_to_f32(h, dtype):
    h = np.ascontiguousarray(h, dtype=np.uint16).ravel()
    out = np.empty(h.size, dtype=np.float32)
    lib().zo_lp_to_f32_array(h.size, _ptr(h, ctypes.c_uint16), _ptr(out, ctypes.c_float), dtype)
    return out


def f32_to_bf16(x):
    return f32_to_lp(x, BF16)


def bf16_to_f32(h):
    return lp_to_f32(h, BF16)


def f32_to_fp16(x):
    return f32_to_lp(x, FP16)


def fp16_to_f32(h):
    return lp_to_f32(h, FP16)


# ------------------------------------------------------------ accounting --
def model_state_bytes(psi, n_d, stage, k=12.0):
    out = (ctypes.c_double * 4)()
    lib().zo_model_state_bytes(float(psi), float(n_d), stage, float(k), out)
    return tuple(out)


def comm_volume(stage):
    return lib().zo_comm_volume(stage)


# ----------------------------------------------------------- collectives --
def all_reduce_mean(grads, dtype, divisor):
    rows = [np.ascontiguousarray(g, dtype=np.uint16) for g in grads]
    psi = rows[0].size
    out = np.empty(psi, dtype=np.float32)
    lib().zo_all_reduce_mean(len(rows), psi, _ptr_array(rows), dtype, divisor, _ptr(out, ctypes.c_float))
    return out


def reduce_scatter(grads, dtype, divisor, shard):
    rows = [np.ascontiguousarray(g, dtype=np.uint16) for g in grads]
    n_d, psi = len(rows), rows[0].size
    out = np.empty(n_d * shard, dtype=np.float32)
    lib().zo_reduce_scatter(n_d, psi, shard, _ptr_array(rows), dtype, divisor,
                            _ptr(out, ctypes.c_float))
    return out


def all_gather_u16(shards, psi, shard):
    rows = [np.ascontiguousarray(s, dtype=np.uint16) for s in shards]
    out = np.zeros(psi, dtype=np.uint16)
    lib().zo_all_gather_u16(len(rows), psi, shard, _ptr_array(rows), _ptr(out, ctypes.c_uint16))
    return out


def all_gather_f32(shards, psi, shard):
    rows = [np.ascontiguousarray(s, dtype=np.float32) for s in shards]
    out = np.zeros(psi, dtype=np.float32)
    lib().zo_all_gather_f32(len(rows), psi, shard, _ptr_array(rows), _ptr(out, ctypes.c_float))
    return out


# ------------------------------------------------------------------ Adam --
def adam_consts(hp, beta1_pow_t, beta2_pow_t):
    c = AdamConsts()
    lib().zo_adam_consts_for(ctypes.byref(hp), beta1_pow_t, beta2_pow_t, ctypes.byref(c))
    return c


def adam_update(hp, consts, g, p, m, v):
    """In-place Adam on float32 arrays p, m, v with gradient g."""
    g = np.ascontiguousarray(g, dtype=np.float32)
    for a in (p, m, v):
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"]
    lib().zo_adam_update(ctypes.byref(hp), ctypes.byref(consts), g.size, _ptr(g, ctypes.c_float),
                         _ptr(p, ctypes.c_float), _ptr(m, ctypes.c_float), _ptr(v, ctypes.c_float))


def sqnorm(g):
    g = np.ascontiguousarray(g, dtype=np.float32)
    return lib().zo_sqnorm(g.size, _ptr(g, ctypes.c_float))


def clip_coef(max_norm, sq):
    applied = ctypes.c_int()
    c = lib().zo_clip_coef(max_norm, sq, ctypes.byref(applied))
    return c, bool(applied.value)


# ------------------------------------------------------------ full steps --
@dataclass
class State:
    """fp32 master / momentum / variance (flat) plus the step scalars."""
    master: np.ndarray
    m: np.ndarray
    v: np.ndarray
    scalars: Scalars = field(default_factory=new_scalars)

    def copy(self):
        sc = Scalars()
        ctypes.memmove(ctypes.byref(sc), ctypes.byref(self.scalars), ctypes.sizeof(Scalars))
        return State(self.master.copy(), self.m.copy(), self.v.copy(), sc)


def plain_dp_step(grads, grad_dtype, hp, state, param_dtype=BF16):
    """All-reduce mean -> full Adam -> cast.  Returns (skipped, params_lp)."""
    rows = [np.ascontiguousarray(g, dtype=np.uint16) for g in grads]
    psi = rows[0].size
    out = np.zeros(psi, dtype=np.uint16)
    skipped = lib().zo_plain_dp_step(len(rows), psi, _ptr_array(rows), grad_dtype, ctypes.byref(hp),
                                     ctypes.byref(state.scalars), _ptr(state.master, ctypes.c_float),
                                     _ptr(state.m, ctypes.c_float), _ptr(state.v, ctypes.c_float),
                                     _ptr(out, ctypes.c_uint16), param_dtype)
    return bool(skipped), out


def zero_step(grads, grad_dtype, hp, state, shard_pad, stage, param_dtype=BF16, lp_shards=None,
              gathered=None):
    """The literal ZeRO path (state arrays are n_d*S long).  Stage 3 writes
    lp_shards (n_d*S), stages 1-2 write gathered (psi).  Returns skipped."""
    rows = [np.ascontiguousarray(g, dtype=np.uint16) for g in grads]
    n_d, psi = len(rows), rows[0].size
    S = shard_size(psi, n_d, shard_pad)
    for a in (state.master, state.m, state.v):
        assert a.size == n_d * S
    if stage >= 3:
        assert lp_shards is not None and lp_shards.size == n_d * S
        lp_p, g_p = _ptr(lp_shards, ctypes.c_uint16), None
    else:
        assert gathered is not None and gathered.size >= psi
        lp_p, g_p = None, _ptr(gathered, ctypes.c_uint16)
    skipped = lib().zo_zero_step(n_d, psi, shard_pad, stage, _ptr_array(rows), grad_dtype,
                                 ctypes.byref(hp), ctypes.byref(state.scalars),
                                 _ptr(state.master, ctypes.c_float), _ptr(state.m, ctypes.c_float),
                                 _ptr(state.v, ctypes.c_float), lp_p, g_p, param_dtype)
    return bool(skipped)


# ---------------------------------------------------- gradient accumulation --
def accumulate_grads(grads, dtype, acc_in=None):
    """acc_out = acc_in (or +0) + the rank-ordered fp32 sum of one
    micro-batch's gradients (not divided).  Returns acc_out (psi fp32)."""
    rows = [np.ascontiguousarray(g, dtype=np.uint16) for g in grads]
    psi = rows[0].size
    out = np.zeros(psi, dtype=np.float32)
    a_in = None if acc_in is None else np.ascontiguousarray(acc_in, dtype=np.float32)
    if a_in is not None:
        assert a_in.size >= psi
    lib().zo_accumulate_grads(len(rows), psi, _ptr_array(rows), dtype,
                              None if a_in is None else _ptr(a_in, ctypes.c_float), _ptr(out, ctypes.c_float))
    return out


def zero_step_accum(grads, grad_dtype, acc, micro, hp, state, shard_pad, stage, param_dtype=BF16,
                    lp_shards=None, gathered=None):
    """The step at the micro-th micro-batch: grads are that micro-batch's
    rank gradients, acc the sum over the earlier ones (None when micro == 1).
    Same outputs as zero_step.  Returns skipped."""
    rows = [np.ascontiguousarray(g, dtype=np.uint16) for g in grads]
    n_d, psi = len(rows), rows[0].size
    S = shard_size(psi, n_d, shard_pad)
    for a in (state.master, state.m, state.v):
        assert a.size == n_d * S
    assert micro >= 1
    a_p = None
    if acc is not None:
        acc = np.ascontiguousarray(acc, dtype=np.float32)
        assert acc.size >= psi
        a_p = _ptr(acc, ctypes.c_float)
    if stage >= 3:
        assert lp_shards is not None and lp_shards.size == n_d * S
        lp_p, g_p = _ptr(lp_shards, ctypes.c_uint16), None
    else:
        assert gathered is not None and gathered.size >= psi
        lp_p, g_p = None, _ptr(gathered, ctypes.c_uint16)
    skipped = lib().zo_zero_step_accum(n_d, psi, shard_pad, stage, _ptr_array(rows), grad_dtype, a_p, micro,
                                       ctypes.byref(hp), ctypes.byref(state.scalars),
                                       _ptr(state.master, ctypes.c_float), _ptr(state.m, ctypes.c_float),
                                       _ptr(state.v, ctypes.c_float), lp_p, g_p, param_dtype)
    return bool(skipped)


# ------------------------------------------------------------- quantizer --
def quantize_block(x_bf16):
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    codes = np.zeros(x.size, dtype=np.int8)
    deq = np.zeros(x.size, dtype=np.uint16)
    scale = ctypes.c_float()
    lib().zo_quantize_block(x.size, _ptr(x, ctypes.c_uint16), _ptr(codes, ctypes.c_int8),
                            ctypes.byref(scale), _ptr(deq, ctypes.c_uint16))
    return codes, scale.value, deq


def quant_gather(shards_flat, n_d, psi, shard, block):
    x = np.ascontiguousarray(shards_flat, dtype=np.uint16)
    assert x.size == n_d * shard
    nbs = (shard + block - 1) // block
    codes = np.zeros(n_d * shard, dtype=np.int8)
    scales = np.zeros(n_d * nbs, dtype=np.float32)
    gathered = np.zeros(psi, dtype=np.uint16)
    lib().zo_quant_gather(n_d, psi, shard, block, _ptr(x, ctypes.c_uint16), _ptr(codes, ctypes.c_int8),
                          _ptr(scales, ctypes.c_float), _ptr(gathered, ctypes.c_uint16))
    return codes, scales, gathered


# ------------------------------------------- quantized gradient exchange --
def qgz_rank_stride(n_d):
    return lib().zo_qgz_rank_stride(n_d)


def quantize_ranks(grads, psi, shard, block):
    """Every rank's int8 codes (psi long, global index) and all scales in one
    array of shape [n_d * nbs, n_dp]: row r * nbs + b, column = rank."""
    rows = [np.ascontiguousarray(g[:psi], dtype=np.uint16) for g in grads]
    n_d = len(rows)
    nbs = (shard + block - 1) // block
    n_dp = qgz_rank_stride(n_d)
    codes = [np.zeros(max(psi, 1), np.int8) for _ in range(n_d)]
    scales = np.zeros((n_d * nbs, n_dp), np.float32)
    lib().zo_quantize_ranks(n_d, psi, shard, block, _ptr_array(rows), _ptr_array(codes), _ptr(scales, ctypes.c_float))
    return codes, scales


def reduce_scatter_q(codes, scales, psi, shard, block, divisor):
    n_d = len(codes)
    out = np.empty(n_d * shard, dtype=np.float32)
    sc = np.ascontiguousarray(scales, dtype=np.float32)
    lib().zo_reduce_scatter_q(n_d, psi, shard, block, _ptr_array(codes), _ptr(sc, ctypes.c_float), divisor,
                              _ptr(out, ctypes.c_float))
    return out


def zero_step_qgz(codes, scales, block, hp, state, shard_pad, stage, psi, param_dtype=BF16, lp_shards=None,
                  gathered=None):
    """The ZeRO step with the quantized gradient exchange (state n_d*S)."""
    n_d = len(codes)
    sc = np.ascontiguousarray(scales, dtype=np.float32)
    if stage >= 3:
        lp_p, g_p = _ptr(lp_shards, ctypes.c_uint16), None
    else:
        lp_p, g_p = None, _ptr(gathered, ctypes.c_uint16)
    return bool(lib().zo_zero_step_qgz(n_d, psi, shard_pad, stage, block, _ptr_array(codes), _ptr(sc, ctypes.c_float),
                                       ctypes.byref(hp), ctypes.byref(state.scalars),
                                       _ptr(state.master, ctypes.c_float), _ptr(state.m, ctypes.c_float),
                                       _ptr(state.v, ctypes.c_float), lp_p, g_p, param_dtype))


def reduce_points_q(codes_at, scales_at, divisor):
    """Reconstructed average at sampled points: codes_at[q], scales_at[q] are
    rank q's codes and block scales gathered at the points."""
    c = [np.ascontiguousarray(x, dtype=np.int8) for x in codes_at]
    sc = [np.ascontiguousarray(x, dtype=np.float32) for x in scales_at]
    out = np.empty(c[0].size, dtype=np.float32)
    lib().zo_reduce_points_q(len(c), c[0].size, _ptr_array(c), _ptr_array(sc), divisor, _ptr(out, ctypes.c_float))
    return out
