"""ctypes binding of libzero.so: one Python function per C entry point, same
names, argument marshalling only.  Every step of the path runs in the CUDA
kernels of the library; nothing here computes.

Device buffers may be passed as torch tensors (their data pointer is used) or
as integer addresses.  ``stream`` defaults to torch's current CUDA stream.
A non-zero status raises ZeroError.  If the library has not been built the
import fails loudly: there is no fallback.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libzero.so")

ZERO_BF16 = 0
ZERO_FP16 = 1
ZERO_MAX_RANKS = 256
ZERO_DEV_TIMEOUT = 1
NOALLOC_SCRATCH_BYTES = 32768 + 4 * (1 << 20)   # ZERO_NOALLOC_SCRATCH_BYTES

STATUS = {0: "ZERO_OK", 1: "ZERO_ERR_INVALID_ARG", 2: "ZERO_ERR_MISALIGNED", 3: "ZERO_ERR_UNSUPPORTED",
          4: "ZERO_ERR_CUDA", 5: "ZERO_ERR_TIMEOUT", 6: "ZERO_ERR_BOUNDS"}


class ZeroError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s failed: %s (%d)" % (where, STATUS.get(status, "?"), status))


class ZeroHparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float), ("max_norm", ctypes.c_float),
                ("loss_scaling", ctypes.c_int), ("scale_window", ctypes.c_int), ("min_scale", ctypes.c_float)]


class ZeroPlanOpts(ctypes.Structure):
    _fields_ = [("param_dtype_set", ctypes.c_int), ("param_dtype", ctypes.c_int),
                ("reduce_bucket_elems", ctypes.c_longlong)]


class ZeroDevScalars(ctypes.Structure):
    _fields_ = [("t", ctypes.c_longlong), ("beta1_pow", ctypes.c_double), ("beta2_pow", ctypes.c_double),
                ("sqnorm", ctypes.c_double), ("loss_scale", ctypes.c_float), ("clip_coef", ctypes.c_float),
                ("good_steps", ctypes.c_int), ("overflow", ctypes.c_int), ("status", ctypes.c_int),
                ("nonfinite", ctypes.c_int), ("ctas_done", ctypes.c_uint), ("reserved", ctypes.c_int)]


if not os.path.exists(LIB_PATH):
    raise ImportError("libzero.so is not built (expected at %s); run "
                      "`python -c \"import __graft_entry__ as g; g.build()\"`" % LIB_PATH)

_lib = ctypes.CDLL(LIB_PATH)

_vp, _ll, _i32, _f32, _f64, _sz = (ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int, ctypes.c_float,
                                   ctypes.c_double, ctypes.c_size_t)
_hp = ctypes.POINTER(ZeroHparams)


class ZeroLayer(ctypes.Structure):
    """zero_layer of zero.h: one layer of the ZeRO-3 layer loop."""
    _fields_ = [("plan", ctypes.c_void_p), ("rank_grads", ctypes.c_void_p), ("acc", ctypes.c_void_p),
                ("master", ctypes.c_void_p), ("m", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("shards_lp", ctypes.c_void_p), ("grads_ready", ctypes.c_void_p), ("stepped", ctypes.c_void_p),
                ("state_on_host", ctypes.c_int)]


_SIGS = {
    "zero_status_str": (ctypes.c_char_p, [_i32]),
    "zero_abi_version": (_i32, []),
    "zero_dev_scalars_size": (_sz, []),
    "zero_plan_create": (_i32, [ctypes.POINTER(_vp), _ll, _i32, _i32, _i32, _i32]),
    "zero_plan_create_ex": (_i32, [ctypes.POINTER(_vp), _ll, _i32, _i32, _i32, _i32,
                                   ctypes.POINTER(ZeroPlanOpts)]),
    "zero_plan_destroy": (None, [_vp]),
    "zero_plan_query": (_i32, [_vp, ctypes.POINTER(_ll), ctypes.POINTER(_ll), ctypes.POINTER(_ll)]),
    "zero_plan_memory": (_i32, [_vp, _i32, _f64, ctypes.POINTER(_f64)]),
    "zero_plan_comm_volume": (_i32, [_vp, _i32, ctypes.POINTER(_f64)]),
    "zero_workspace_bytes": (_sz, [_vp, _hp]),
    "zero_scalars_init": (_i32, [_vp, _f32, _vp]),
    "zero_reduce_scatter": (_i32, [_vp, _vp, _hp, _vp, _vp, _vp, _vp]),
    "zero_grad_sqnorm": (_i32, [_vp, _vp, _hp, _vp, _vp, _vp]),
    "zero_adam_shard_step": (_i32, [_vp, _hp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "zero_all_gather": (_i32, [_vp, _vp, _vp, _vp, _vp]),
    "zero_step_fused": (_i32, [_vp, _hp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "zero_quant_gather": (_i32, [_vp, _vp, _i32, _vp, _vp, _vp, _vp]),
    "zero_step_fused_qgather": (_i32, [_vp, _hp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _vp,
                                       _vp, _vp, _vp]),
    "zero_debug_wait_timeout": (_i32, [_vp, _ll, _vp]),
    "zero_debug_stream_timeout": (_i32, [_i32, _vp, _vp, _ll, _vp]),
    "zero_launch_count": (ctypes.c_ulonglong, []),
    "zero_step_fused_noalloc": (_i32, [_vp, _hp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "zero_quantize_grads": (_i32, [_vp, _vp, _i32, _vp, _vp, _vp, _vp]),
    "zero_step_fused_offload": (_i32, [_vp, _hp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "zero_accumulate_grads": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp]),
    "zero_step_fused_accum": (_i32, [_vp, _hp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "zero_step_fused_qgz": (_i32, [_vp, _hp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "zero_step_fused_qgz_qgather": (_i32, [_vp, _hp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                           _vp, _vp, _vp]),
    "zero_step_layers": (_i32, [_hp, _i32, ctypes.POINTER(ZeroLayer), _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp,
                                _vp]),
    "zero_layers_workspace_bytes": (_sz, [_hp, _i32, ctypes.POINTER(ZeroLayer)]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


# ----------------------------------------------------------------- marshalling
def _addr(x):
    """Device address of a torch tensor, an int, or None (NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def rank_ptrs(bufs):
    """The host array of device pointers that the entry points taking one
    buffer per rank read, built once.  Any call accepts it in place of a list
    of tensors, which saves marshalling the list on every call (a few
    microseconds, the whole launch cost of a small step).  It holds addresses
    only: the caller keeps the tensors alive and in place."""
    arr = (ctypes.c_void_p * len(bufs))()
    for i, b in enumerate(bufs):
        arr[i] = _addr(b)
    return arr


def _ptr_array(bufs):
    if isinstance(bufs, ctypes.Array):
        return bufs
    return rank_ptrs(bufs)


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status, where):
    if status != 0:
        raise ZeroError(status, where)


def hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, max_norm=0.0, loss_scaling=False,
            scale_window=1000, min_scale=1.0):
    return ZeroHparams(lr, beta1, beta2, eps, weight_decay, max_norm, int(bool(loss_scaling)), scale_window,
                       min_scale)


# ------------------------------------------------------------- entry points
def zero_status_str(status):
    return _lib.zero_status_str(status).decode()


def zero_abi_version():
    return _lib.zero_abi_version()


def zero_dev_scalars_size():
    return _lib.zero_dev_scalars_size()


def zero_plan_create(psi, n_d, stage, grad_dtype, shard_pad):
    h = ctypes.c_void_p()
    _check(_lib.zero_plan_create(ctypes.byref(h), psi, n_d, stage, grad_dtype, shard_pad), "zero_plan_create")
    return h


def zero_plan_create_ex(psi, n_d, stage, grad_dtype, shard_pad, param_dtype=None, reduce_bucket_elems=0):
    h = ctypes.c_void_p()
    opts = ZeroPlanOpts(0 if param_dtype is None else 1, 0 if param_dtype is None else param_dtype,
                        reduce_bucket_elems)
    _check(_lib.zero_plan_create_ex(ctypes.byref(h), psi, n_d, stage, grad_dtype, shard_pad, ctypes.byref(opts)),
           "zero_plan_create_ex")
    return h


def zero_plan_destroy(plan):
    _lib.zero_plan_destroy(plan)


def zero_plan_query(plan, n_d):
    s, p = ctypes.c_longlong(), ctypes.c_longlong()
    lens = (ctypes.c_longlong * n_d)()
    _check(_lib.zero_plan_query(plan, ctypes.byref(s), ctypes.byref(p), lens), "zero_plan_query")
    return s.value, p.value, list(lens)


def zero_plan_memory(plan, stage, k=12.0):
    out = (ctypes.c_double * 4)()
    _check(_lib.zero_plan_memory(plan, stage, k, out), "zero_plan_memory")
    return tuple(out)


def zero_plan_comm_volume(plan, stage):
    out = ctypes.c_double()
    _check(_lib.zero_plan_comm_volume(plan, stage, ctypes.byref(out)), "zero_plan_comm_volume")
    return out.value


def zero_workspace_bytes(plan, hp):
    return _lib.zero_workspace_bytes(plan, ctypes.byref(hp) if hp is not None else None)


def zero_scalars_init(scalars, loss_scale=1.0, stream=None):
    _check(_lib.zero_scalars_init(_addr(scalars), loss_scale, _stream(stream)), "zero_scalars_init")


def zero_reduce_scatter(plan, rank_grads, hp, scalars, grad_shards, ws, stream=None):
    _check(_lib.zero_reduce_scatter(plan, _ptr_array(rank_grads), ctypes.byref(hp), _addr(scalars),
                                    _addr(grad_shards), _addr(ws), _stream(stream)), "zero_reduce_scatter")


def zero_grad_sqnorm(plan, grad_shards, hp, scalars, ws, stream=None):
    _check(_lib.zero_grad_sqnorm(plan, _addr(grad_shards), ctypes.byref(hp), _addr(scalars), _addr(ws),
                                 _stream(stream)), "zero_grad_sqnorm")


def zero_adam_shard_step(plan, hp, grad_shards, master, m, v, lp_out, scalars, stream=None):
    _check(_lib.zero_adam_shard_step(plan, ctypes.byref(hp), _addr(grad_shards), _addr(master), _addr(m),
                                     _addr(v), _addr(lp_out), _addr(scalars), _stream(stream)),
           "zero_adam_shard_step")


def zero_all_gather(plan, shards_lp, gathered, scalars=None, stream=None):
    _check(_lib.zero_all_gather(plan, _ptr_array(shards_lp), _addr(gathered), _addr(scalars), _stream(stream)),
           "zero_all_gather")


def zero_step_fused(plan, hp, rank_grads, master_in, m_in, v_in, master_out, m_out, v_out, lp_out, scalars, ws,
                    stream=None):
    _check(_lib.zero_step_fused(plan, ctypes.byref(hp), _ptr_array(rank_grads), _addr(master_in), _addr(m_in),
                                _addr(v_in), _addr(master_out), _addr(m_out), _addr(v_out), _addr(lp_out),
                                _addr(scalars), _addr(ws), _stream(stream)), "zero_step_fused")


def zero_step_fused_offload(plan, hp, rank_grads, master_in, m_in, v_in, master_out, m_out, v_out, lp_out, scalars,
                            ws, stream=None):
    """zero_step_fused with master/m/v in page-locked host memory (pin_memory tensors)."""
    _check(_lib.zero_step_fused_offload(plan, ctypes.byref(hp), _ptr_array(rank_grads), _addr(master_in),
                                        _addr(m_in), _addr(v_in), _addr(master_out), _addr(m_out), _addr(v_out),
                                        _addr(lp_out), _addr(scalars), _addr(ws), _stream(stream)),
           "zero_step_fused_offload")


def zero_accumulate_grads(plan, rank_grads, acc_in, acc_out, scalars=None, stream=None):
    """acc_out = acc_in (None: +0) + this micro-batch's rank sum (fp32, undivided)."""
    _check(_lib.zero_accumulate_grads(plan, _ptr_array(rank_grads), _addr(acc_in), _addr(acc_out), _addr(scalars),
                                      _stream(stream)), "zero_accumulate_grads")


def zero_step_fused_accum(plan, hp, rank_grads, acc, micro_batches, master_in, m_in, v_in, master_out, m_out, v_out,
                          lp_out, scalars, ws, stream=None):
    """The step at the last of micro_batches micro-batches (acc: sum of the earlier ones, None when 1)."""
    _check(_lib.zero_step_fused_accum(plan, ctypes.byref(hp), _ptr_array(rank_grads), _addr(acc), micro_batches,
                                      _addr(master_in), _addr(m_in), _addr(v_in), _addr(master_out), _addr(m_out),
                                      _addr(v_out), _addr(lp_out), _addr(scalars), _addr(ws), _stream(stream)),
           "zero_step_fused_accum")


def zero_quant_gather(plan, shards_bf16, block, codes, scales, gathered, stream=None):
    _check(_lib.zero_quant_gather(plan, _addr(shards_bf16), block, _addr(codes), _addr(scales), _addr(gathered),
                                  _stream(stream)), "zero_quant_gather")


def zero_step_fused_qgather(plan, hp, rank_grads, master_in, m_in, v_in, master_out, m_out, v_out, block, codes,
                            scales, gathered, scalars, ws, stream=None):
    _check(_lib.zero_step_fused_qgather(plan, ctypes.byref(hp), _ptr_array(rank_grads), _addr(master_in),
                                        _addr(m_in), _addr(v_in), _addr(master_out), _addr(m_out), _addr(v_out),
                                        block, _addr(codes), _addr(scales), _addr(gathered), _addr(scalars),
                                        _addr(ws), _stream(stream)), "zero_step_fused_qgather")


def zero_quantize_grads(plan, rank_grads, block, rank_codes, rank_scales, scalars=None, stream=None):
    _check(_lib.zero_quantize_grads(plan, _ptr_array(rank_grads), block, _ptr_array(rank_codes),
                                    _addr(rank_scales), _addr(scalars), _stream(stream)), "zero_quantize_grads")


def zero_step_fused_qgz(plan, hp, rank_codes, rank_scales, block, master_in, m_in, v_in, master_out, m_out, v_out,
                        lp_out, scalars, ws=None, stream=None):
    """ws: the workspace, needed with clipping (None otherwise)."""
    _check(_lib.zero_step_fused_qgz(plan, ctypes.byref(hp), _ptr_array(rank_codes), _addr(rank_scales), block,
                                    _addr(master_in), _addr(m_in), _addr(v_in), _addr(master_out), _addr(m_out),
                                    _addr(v_out), _addr(lp_out), _addr(scalars), _addr(ws), _stream(stream)),
           "zero_step_fused_qgz")


def zero_step_fused_qgz_qgather(plan, hp, rank_codes, rank_scales, block, master_in, m_in, v_in, master_out, m_out,
                                v_out, codes_out, scales_out, gathered, scalars, ws=None, stream=None):
    """Both ZeRO++ exchanges in one step: int8 rank codes in, int8 gather out
    (ws: the workspace, needed with clipping)."""
    _check(_lib.zero_step_fused_qgz_qgather(plan, ctypes.byref(hp), _ptr_array(rank_codes), _addr(rank_scales),
                                            block, _addr(master_in), _addr(m_in), _addr(v_in), _addr(master_out),
                                            _addr(m_out), _addr(v_out), _addr(codes_out), _addr(scales_out),
                                            _addr(gathered), _addr(scalars), _addr(ws), _stream(stream)),
           "zero_step_fused_qgz_qgather")


def zero_debug_wait_timeout(scalars, timeout_ns, stream=None):
    _check(_lib.zero_debug_wait_timeout(_addr(scalars), timeout_ns, _stream(stream)), "zero_debug_wait_timeout")


def zero_debug_stream_timeout(kernel, scratch, scalars, timeout_ns, stream=None):
    """One launch of a pipelined kernel (0 engine, 1 all-gather, 2 sender)
    whose bulk copies are never issued: every wait runs out (tests the timeout path)."""
    _check(_lib.zero_debug_stream_timeout(kernel, _addr(scratch), _addr(scalars), timeout_ns, _stream(stream)),
           "zero_debug_stream_timeout")


def zero_step_fused_noalloc(plan, hp, rank_grads, master_in, m_in, v_in, master_out, m_out, v_out, lp_out,
                            scalars, stream=None):
    """zero_step_fused without a workspace argument, for callers that cannot
    allocate device memory: the library's own scratch array of
    NOALLOC_SCRATCH_BYTES serves as the workspace.  Its limit (clipping with
    n_d > 4 needs n_d*S <= 2^20), its set-up (the first call on a device, and
    after a device reset, looks up the array's address: make it before any
    stream capture) and its sharing rule (overlapping calls race on the one
    array) are stated in include/zero.h."""
    _check(_lib.zero_step_fused_noalloc(plan, ctypes.byref(hp), _ptr_array(rank_grads), _addr(master_in),
                                        _addr(m_in), _addr(v_in), _addr(master_out), _addr(m_out), _addr(v_out),
                                        _addr(lp_out), _addr(scalars), _stream(stream)),
           "zero_step_fused_noalloc")


def _event(ev):
    """cudaEvent_t of a torch.cuda.Event (recorded once if torch has not
    created it yet), an int handle, or None."""
    if ev is None or isinstance(ev, int):
        return ev
    if not ev.cuda_event:
        ev.record()
    return ev.cuda_event


class LayerStack:
    """The zero_layer array of a stack of layers, built once (the pointers it
    holds stay valid while the caller keeps the tensors alive and in place).
    layers: sequence of (plan_handle, rank_grads, master, m, v, shards_lp
    [, grads_ready, stepped[, acc[, state_on_host]]]), rank_grads a list of
    per-rank tensors or a rank_ptrs array, the two events torch.cuda.Event
    objects or None, acc the layer's accumulated earlier micro-batches or
    None, state_on_host True when master/m/v are page-locked host tensors."""

    def __init__(self, layers):
        self._ranks = [_ptr_array(l[1]) for l in layers]
        self.array = (ZeroLayer * len(layers))()
        for i, l in enumerate(layers):
            plan, _, master, m, v, shards = l[:6]
            ready, stepped, acc, host = (tuple(l[6:10]) + (None, None, None, False))[:4]
            self.array[i] = ZeroLayer(plan, ctypes.cast(self._ranks[i], ctypes.c_void_p), _addr(acc), _addr(master),
                                      _addr(m), _addr(v), _addr(shards), _event(ready), _event(stepped), int(bool(host)))

    def __len__(self):
        return len(self.array)


def _stack(layers):
    return layers if isinstance(layers, LayerStack) else LayerStack(layers)


def zero_layers_workspace_bytes(hp, layers):
    stack = _stack(layers)
    return _lib.zero_layers_workspace_bytes(ctypes.byref(hp), len(stack), stack.array)


def zero_step_layers(hp, layers, gathers, gathered, scalars, ws=None, micro_batches=1, stream=None,
                     gather_stream=None, gathered_codes=None, gathered_scales=None):
    """One ZeRO-3 step over a stack of layers: layer l's gather(s) into
    gathered[l % len(gathered)], then its fused step; with gather_stream the
    gathers run there, the next layer's overlapping this layer's step.  With
    clipping or loss scaling the global checks span every layer (ws: see
    zero_layers_workspace_bytes).  With gathered_codes / gathered_scales (one
    per gathered buffer) the gathers are block-int8 quantized (qwZ).
    layers: a LayerStack (or the sequence it is built from)."""
    stack = _stack(layers)
    gptr = _ptr_array(gathered)
    cptr = None if gathered_codes is None else _ptr_array(gathered_codes)
    sptr = None if gathered_scales is None else _ptr_array(gathered_scales)
    gs = None if gather_stream is None else _stream(gather_stream)
    _check(_lib.zero_step_layers(ctypes.byref(hp), len(stack), stack.array, micro_batches, gathers, len(gptr), gptr,
                                 cptr, sptr, _addr(scalars), _addr(ws), _stream(stream), gs), "zero_step_layers")


def zero_launch_count():
    return _lib.zero_launch_count()


def raw_status(call, *args):
    """Call an entry point by name with raw ctypes arguments and return its
    status instead of raising (for argument-checking tests)."""
    return getattr(_lib, call)(*args)


def library():
    return _lib
