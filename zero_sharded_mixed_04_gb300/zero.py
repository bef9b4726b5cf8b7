"""ctypes binding of libzero_gb300.so (declared in include/zero_gb300.h).

The functions have the C names and argument order.  This module only
marshals arguments.  Device buffers may be given as torch tensors (their
``data_ptr()`` is passed) or as integer addresses.  Status codes come back as
the C functions return them; ``check()`` turns a negative one into an
exception.

Importing this module loads the shared library.  If it has not been built
(``python -m zero_sharded_mixed_04_gb300.build``), the import raises
ImportError: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
# ZERO_GB300_DEBUG=1 loads the debug build (device-side bounds checks) instead
DEBUG_BUILD = os.environ.get("ZERO_GB300_DEBUG", "") not in ("", "0")
LIB_PATH = os.path.join(_PKG, "libzero_gb300_debug.so" if DEBUG_BUILD else "libzero_gb300.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -m zero_sharded_mixed_04_gb300.build` "
        "(or __graft_entry__.build()); the ZeRO step has no non-CUDA implementation")

_lib = ctypes.CDLL(LIB_PATH)

ZERO_PAD_UNIT = 128
ZERO_MAX_RANKS = 64
ZERO_ALIGN_BYTES = 16
ZERO_BUCKET_ALIGN = 8
ZERO_MAX_ELEMS = 1 << 48

ZERO_OK = 0
ZERO_STEP_SKIPPED = 1
ZERO_ERR_ARG = -1
ZERO_ERR_ALIGN = -2
ZERO_ERR_CUDA = -3
ZERO_ERR_TIMEOUT = -4
ZERO_ERR_WORKSPACE = -5
ZERO_ERR_OVERLAP = -6
ZERO_ERR_TOO_LARGE = -7
ZERO_ERR_POLICY_WINDOW = -8
ZERO_ERR_BOUNDS = -9
ZERO_POLICY_WINDOW = 16

ZERO_WORKSPACE_CONTROL_BYTES = 16640
ZERO_NOALLOC_MAX_TWO_PASS_ELEMS = 4194304
ZERO_NOALLOC_SCRATCH_BYTES = 16640 + 4 * ZERO_NOALLOC_MAX_TWO_PASS_ELEMS

ZERO_GRAD_BF16 = 0
ZERO_GRAD_FP32 = 1

ZERO_STAGING_REGISTERS = 0
ZERO_STAGING_TMA = 1
ZERO_STAGING_TMA_TEST_STALL = 2

ZERO3_GATHER_OVERLAP_PREVIOUS = 1


class zero_layout(ctypes.Structure):
    _fields_ = [("psi", ctypes.c_int64), ("psi_pad", ctypes.c_int64), ("shard", ctypes.c_int64),
                ("n_tensors", ctypes.c_int64), ("N", ctypes.c_int32), ("pad_unit", ctypes.c_int32)]


class zero_adam_hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double),
                ("max_grad_norm", ctypes.c_double), ("step", ctypes.c_int64),
                ("skip_on_overflow", ctypes.c_int32), ("micro_batches", ctypes.c_int32),
                ("bucket_elems", ctypes.c_int64)]


class zero_step_result(ctypes.Structure):
    _fields_ = [("status", ctypes.c_int32), ("found_nonfinite", ctypes.c_uint32),
                ("grad_norm", ctypes.c_float), ("clip_coef", ctypes.c_float)]


class zero_plan(ctypes.Structure):
    _fields_ = [("grads", ctypes.c_void_p * ZERO_MAX_RANKS), ("src_master", ctypes.c_void_p),
                ("src_m", ctypes.c_void_p), ("src_v", ctypes.c_void_p),
                ("src_w_bf16", ctypes.c_void_p), ("dst_master", ctypes.c_void_p),
                ("dst_m", ctypes.c_void_p), ("dst_v", ctypes.c_void_p),
                ("dst_w_bf16", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("grad_accum", ctypes.c_void_p),
                ("psi_pad", ctypes.c_int64),
                ("cursor", ctypes.c_int64), ("hp", zero_adam_hparams),
                ("loss_scale", ctypes.c_float), ("grad_dtype", ctypes.c_int32),
                ("N", ctypes.c_int32), ("in_place", ctypes.c_int32), ("two_pass", ctypes.c_int32),
                ("state", ctypes.c_int32), ("micro_batch", ctypes.c_int32),
                ("policy_t_count", ctypes.c_int32), ("policy_t_first", ctypes.c_int64),
                ("policy", ctypes.c_void_p), ("overlap_buckets", ctypes.c_int32),
                ("smem_staging", ctypes.c_int32), ("current_set", ctypes.c_void_p),
                ("rows_offset", ctypes.c_int64), ("row_capacity", ctypes.c_int32),
                ("rows_used", ctypes.c_int32), ("row_width", ctypes.c_int32),
                ("shared_slots_used", ctypes.c_int32),
                ("policy_table", ctypes.c_void_p)]


class zero_device_policy(ctypes.Structure):
    _fields_ = [("t", ctypes.c_int64), ("loss_scale", ctypes.c_float),
                ("good_steps", ctypes.c_int32), ("growth_interval", ctypes.c_int32),
                ("backoff", ctypes.c_float), ("growth", ctypes.c_float),
                ("last_status", ctypes.c_int32)]


_P = ctypes.c_void_p
_i32, _i64, _f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float
_PLAN = ctypes.POINTER(zero_plan)

_lib.zero_init_layout.argtypes = [_P, _i64, _i32, ctypes.POINTER(zero_layout), _P]
_lib.zero_init_layout.restype = ctypes.c_int
_lib.zero_shard_range.argtypes = [ctypes.POINTER(zero_layout), _i32, ctypes.POINTER(_i64),
                                  ctypes.POINTER(_i64)]
_lib.zero_shard_range.restype = ctypes.c_int
_lib.zero_workspace_bytes.argtypes = [_i64, ctypes.POINTER(zero_adam_hparams), _i32]
_lib.zero_workspace_bytes.restype = ctypes.c_size_t
_lib.zero_step.argtypes = [_P, _i32, _P, _P, _P, _P, _i64, _i32,
                           ctypes.POINTER(zero_adam_hparams), _f32, _P, ctypes.c_size_t, _P, _P]
_lib.zero_step.restype = ctypes.c_int
_lib.zero_step_into.argtypes = [_P, _i32, _P, _P, _P, _P, _P, _P, _P, _P, _i64, _i32,
                                ctypes.POINTER(zero_adam_hparams), _f32, _P, ctypes.c_size_t,
                                _P, _P]
_lib.zero_step_into.restype = ctypes.c_int
_lib.zero_plan_init.argtypes = [_PLAN, _P, _i32, _P, _P, _P, _P, _P, _P, _P, _P, _i64, _i32,
                                ctypes.POINTER(zero_adam_hparams), _f32, _P, ctypes.c_size_t]
_lib.zero_plan_init.restype = ctypes.c_int
_lib.zero_plan_init_ex.argtypes = [_PLAN, _P, _i32, _P, _P, _P, _P, _P, _P, _P, _P, _i64, _i32,
                                   ctypes.POINTER(zero_adam_hparams), _f32, _P, ctypes.c_size_t, _P]
_lib.zero_plan_init_ex.restype = ctypes.c_int
_lib.zero_plan_set_device_policy.argtypes = [_PLAN, _P, _i64, _i32]
_lib.zero_plan_set_device_policy.restype = ctypes.c_int
_lib.zero_policy_table_fill.argtypes = [ctypes.POINTER(zero_adam_hparams), _i64, _i64, _P]
_lib.zero_policy_table_fill.restype = ctypes.c_int
_lib.zero_plan_set_device_policy_table.argtypes = [_PLAN, _P, _P, _i64, _i32]
_lib.zero_plan_set_device_policy_table.restype = ctypes.c_int
_lib.zero_plan_set_pingpong.argtypes = [_PLAN, _P]
_lib.zero_plan_set_pingpong.restype = ctypes.c_int
_lib.zero_plan_begin.argtypes = [_PLAN, _P]
_lib.zero_plan_begin.restype = ctypes.c_int
_lib.zero_plan_bucket.argtypes = [_PLAN, _i64, _i64, _P, _P]
_lib.zero_plan_bucket.restype = ctypes.c_int
_lib.zero_plan_end.argtypes = [_PLAN, _P, _P]
_lib.zero_plan_end.restype = ctypes.c_int
_lib.zero_step_noalloc.argtypes = [_P, _i32, _P, _P, _P, _P, _i64, _i32,
                                   ctypes.POINTER(zero_adam_hparams), _f32, _P, _P]
_lib.zero_step_noalloc.restype = ctypes.c_int
_lib.zero3_gather.argtypes = [_P, _i32, _i64, _i64, _i64, _P, ctypes.c_uint32, _P]
_lib.zero3_gather.restype = ctypes.c_int
_lib.zero3_peak_bytes.argtypes = [_P, _i64, _i32, _i32, _i32]
_lib.zero3_peak_bytes.restype = _i64
_lib.zero_ledger.argtypes = [_i64, _i32, _i32, _i32, _i32]
_lib.zero_ledger.restype = _i64
_lib.zero_comm_volume.argtypes = [_i64, _i32, _i32]
_lib.zero_comm_volume.restype = _i64
_lib.zero_status_str.argtypes = [ctypes.c_int]
_lib.zero_status_str.restype = ctypes.c_char_p
_lib.zero_launch_count.argtypes = []
_lib.zero_launch_count.restype = ctypes.c_uint64
_lib.zero_debug_bounds_violations.argtypes = []
_lib.zero_debug_bounds_violations.restype = ctypes.c_int64


class ZeroError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {zero_status_str(status)} ({status})" if what
                         else f"{zero_status_str(status)} ({status})")


def check(status: int, what: str = "") -> int:
    """Raise ZeroError for a negative status; return it otherwise."""
    if status < 0:
        raise ZeroError(status, what)
    return status


def _addr(x) -> int | None:
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr() if x.numel() > 0 else None
    if isinstance(x, ctypes.Structure):
        return ctypes.addressof(x)
    return int(x)


def _stream(s) -> int | None:
    """None -> torch's current CUDA stream; a torch stream -> its handle; an int
    -> that handle (0 is the legacy default stream)."""
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream or None
    return int(s) or None


def make_hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0,
                 max_grad_norm=0.0, step=1, skip_on_overflow=False,
                 bucket_elems=0, micro_batches=0) -> zero_adam_hparams:
    return zero_adam_hparams(lr, beta1, beta2, eps, weight_decay, max_grad_norm, step,
                             int(bool(skip_on_overflow)), micro_batches, bucket_elems)


def zero_init_layout(tensor_numel, N: int):
    """Returns (status, zero_layout, offsets list)."""
    n = len(tensor_numel)
    arr = (ctypes.c_int64 * max(n, 1))(*[int(x) for x in tensor_numel])
    offs = (ctypes.c_int64 * max(n, 1))()
    lay = zero_layout()
    rc = _lib.zero_init_layout(arr if n else None, n, N, ctypes.byref(lay), offs)
    return rc, lay, [offs[i] for i in range(n)]


def zero_shard_range(layout: zero_layout, r: int):
    """Returns (status, begin, end)."""
    b, e = ctypes.c_int64(), ctypes.c_int64()
    rc = _lib.zero_shard_range(ctypes.byref(layout), r, ctypes.byref(b), ctypes.byref(e))
    return rc, b.value, e.value


def zero_workspace_bytes(psi_pad: int, hp: zero_adam_hparams, in_place: bool) -> int:
    return _lib.zero_workspace_bytes(psi_pad, ctypes.byref(hp), int(bool(in_place)))


def _grad_array(grads, N=None):
    """The C array of gradient pointers, padded with NULLs to N entries: a list
    shorter than N reaches the library as missing gradients (an argument error),
    never as a read past the end of the array."""
    n = len(grads)
    if N is not None:
        n = max(n, min(max(int(N), 0), ZERO_MAX_RANKS))
    ptrs = [_addr(g) for g in grads] + [None] * (n - len(grads))
    return (ctypes.c_void_p * max(n, 1))(*ptrs)


def _check(x, nbytes: int, name: str) -> None:
    """A torch tensor handed over as a buffer must be contiguous and hold the
    nbytes the call will touch.  Raw addresses are the caller's to size."""
    if x is None or not hasattr(x, "data_ptr") or nbytes <= 0:
        return
    if not x.is_contiguous():
        raise ValueError(f"{name}: the tensor is not contiguous")
    have = x.numel() * x.element_size()
    if have < nbytes:
        raise ValueError(f"{name}: the tensor holds {have} bytes, the call uses {nbytes}")


def _check_step(grads, grad_dtype: int, psi_pad: int, state, workspace=None,
                workspace_bytes: int = 0) -> None:
    """The sizes a step reads and writes: N gradients of psi_pad elements,
    FP32 master/m/v and BF16 weights of psi_pad elements, the workspace."""
    if not 0 < psi_pad <= ZERO_MAX_ELEMS:
        return  # sizes the library refuses are left for it to refuse
    g = 2 if grad_dtype == ZERO_GRAD_BF16 else 4
    for i, t in enumerate(grads):
        _check(t, psi_pad * g, f"grads[{i}]")
    for name, t, elem in state:
        _check(t, psi_pad * elem, name)
    _check(workspace, workspace_bytes, "workspace")


def _state(prefix, master, m, v, w):
    return [(prefix + "master", master, 4), (prefix + "m", m, 4), (prefix + "v", v, 4),
            (prefix + "w_bf16", w, 2)]


def zero_step(grads, grad_dtype: int, master, m, v, w_bf16, psi_pad: int, N: int,
              hp: zero_adam_hparams, loss_scale: float, workspace, workspace_bytes: int,
              result=None, stream=None) -> int:
    _check_step(grads, grad_dtype, psi_pad, _state("", master, m, v, w_bf16), workspace,
                workspace_bytes)
    _check(result, 16, "result")
    return _lib.zero_step(_grad_array(grads, N), grad_dtype, _addr(master), _addr(m), _addr(v),
                          _addr(w_bf16), psi_pad, N, ctypes.byref(hp), loss_scale,
                          _addr(workspace), workspace_bytes, _addr(result), _stream(stream))


def zero_step_into(grads, grad_dtype: int, src_master, src_m, src_v, src_w_bf16, dst_master,
                   dst_m, dst_v, dst_w_bf16, psi_pad: int, N: int, hp: zero_adam_hparams,
                   loss_scale: float, workspace, workspace_bytes: int, result=None,
                   stream=None) -> int:
    _check_step(grads, grad_dtype, psi_pad,
                _state("src_", src_master, src_m, src_v, src_w_bf16) +
                _state("dst_", dst_master, dst_m, dst_v, dst_w_bf16), workspace, workspace_bytes)
    _check(result, 16, "result")
    return _lib.zero_step_into(_grad_array(grads, N), grad_dtype, _addr(src_master), _addr(src_m),
                               _addr(src_v), _addr(src_w_bf16), _addr(dst_master), _addr(dst_m),
                               _addr(dst_v), _addr(dst_w_bf16), psi_pad, N, ctypes.byref(hp),
                               loss_scale, _addr(workspace), workspace_bytes, _addr(result),
                               _stream(stream))


def zero_plan_init(plan: zero_plan, grads, grad_dtype: int, src_master, src_m, src_v, src_w_bf16,
                   dst_master, dst_m, dst_v, dst_w_bf16, psi_pad: int, N: int,
                   hp: zero_adam_hparams, loss_scale: float, workspace,
                   workspace_bytes: int) -> int:
    _check_step(grads, grad_dtype, psi_pad,
                _state("src_", src_master, src_m, src_v, src_w_bf16) +
                _state("dst_", dst_master, dst_m, dst_v, dst_w_bf16), workspace, workspace_bytes)
    return _lib.zero_plan_init(ctypes.byref(plan), _grad_array(grads, N), grad_dtype,
                               _addr(src_master), _addr(src_m), _addr(src_v), _addr(src_w_bf16),
                               _addr(dst_master), _addr(dst_m), _addr(dst_v), _addr(dst_w_bf16),
                               psi_pad, N, ctypes.byref(hp), loss_scale, _addr(workspace),
                               workspace_bytes)


def zero_plan_init_ex(plan: zero_plan, grads, grad_dtype: int, src_master, src_m, src_v,
                      src_w_bf16, dst_master, dst_m, dst_v, dst_w_bf16, psi_pad: int, N: int,
                      hp: zero_adam_hparams, loss_scale: float, workspace, workspace_bytes: int,
                      grad_accum=None) -> int:
    _check_step(grads, grad_dtype, psi_pad,
                _state("src_", src_master, src_m, src_v, src_w_bf16) +
                _state("dst_", dst_master, dst_m, dst_v, dst_w_bf16) +
                [("grad_accum", grad_accum, 4)], workspace, workspace_bytes)
    return _lib.zero_plan_init_ex(ctypes.byref(plan), _grad_array(grads, N), grad_dtype,
                                  _addr(src_master), _addr(src_m), _addr(src_v),
                                  _addr(src_w_bf16), _addr(dst_master), _addr(dst_m),
                                  _addr(dst_v), _addr(dst_w_bf16), psi_pad, N, ctypes.byref(hp),
                                  loss_scale, _addr(workspace), workspace_bytes,
                                  _addr(grad_accum))


def zero_plan_set_device_policy(plan: zero_plan, policy, t_first: int, t_count: int) -> int:
    """policy: the address of a device-addressable zero_device_policy (a pinned
    host tensor or device tensor of its size)."""
    return _lib.zero_plan_set_device_policy(ctypes.byref(plan), _addr(policy), t_first, t_count)


def zero_policy_table_fill(hp: zero_adam_hparams, t_first: int, t_count: int, table) -> int:
    """table: a host buffer of 2 * t_count floats (a CPU tensor or an address)."""
    if t_count > 0:
        _check(table, 8 * t_count, "table")
    return _lib.zero_policy_table_fill(ctypes.byref(hp), t_first, t_count, _addr(table))


def zero_plan_set_device_policy_table(plan: zero_plan, policy, table, t_first: int,
                                      t_count: int) -> int:
    """policy as for zero_plan_set_device_policy; table: a device-addressable
    buffer of 2 * t_count floats filled by zero_policy_table_fill."""
    if t_count > 0:
        _check(table, 8 * t_count, "table")
    return _lib.zero_plan_set_device_policy_table(ctypes.byref(plan), _addr(policy), _addr(table),
                                                  t_first, t_count)


def zero_plan_set_pingpong(plan: zero_plan, current_set) -> int:
    """current_set: the address of a device-addressable int32 (a pinned host
    tensor or a device tensor) naming the current state set, 0 or 1."""
    return _lib.zero_plan_set_pingpong(ctypes.byref(plan), _addr(current_set))


def zero_plan_begin(plan: zero_plan, stream=None) -> int:
    return _lib.zero_plan_begin(ctypes.byref(plan), _stream(stream))


def zero_plan_bucket(plan: zero_plan, begin: int, end: int, bucket_grads=None,
                     stream=None) -> int:
    arr = None
    if bucket_grads is not None:
        g = 2 if plan.grad_dtype == ZERO_GRAD_BF16 else 4
        if 0 <= begin < end <= plan.psi_pad:
            for i, t in enumerate(bucket_grads):
                _check(t, (end - begin) * g, f"bucket_grads[{i}]")
        arr = _grad_array(bucket_grads, plan.N)
    return _lib.zero_plan_bucket(ctypes.byref(plan), begin, end, arr, _stream(stream))


def zero_plan_end(plan: zero_plan, result=None, stream=None) -> int:
    _check(result, 16, "result")
    return _lib.zero_plan_end(ctypes.byref(plan), _addr(result), _stream(stream))


def zero_step_noalloc(grads, grad_dtype: int, master, m, v, w_bf16, psi_pad: int, N: int,
                      hp: zero_adam_hparams, loss_scale: float, result=None,
                      stream=None) -> int:
    """zero_step with the library's fixed scratch array as its workspace, for
    callers that cannot allocate device memory (see include/zero_gb300.h)."""
    _check_step(grads, grad_dtype, psi_pad, _state("", master, m, v, w_bf16))
    _check(result, 16, "result")
    return _lib.zero_step_noalloc(_grad_array(grads, N), grad_dtype, _addr(master), _addr(m),
                                  _addr(v), _addr(w_bf16), psi_pad, N, ctypes.byref(hp),
                                  loss_scale, _addr(result), _stream(stream))


def zero3_gather(shards, N: int, shard: int, begin: int, end: int, view, stream=None,
                 flags: int = 0) -> int:
    """Elements [begin, end) of the full BF16 view, gathered from N shards."""
    # sizes the library refuses are left for it to refuse
    if 1 <= N <= ZERO_MAX_RANKS and 0 < shard <= ZERO_MAX_ELEMS // N and 0 <= begin < end <= N * shard:
        for i, t in enumerate(shards):
            _check(t, 2 * shard, f"shards[{i}]")
        _check(view, 2 * (end - begin), "view")
    arr = _grad_array(shards, N)
    return _lib.zero3_gather(arr, N, shard, begin, end, _addr(view), flags, _stream(stream))


def zero3_peak_bytes(layer_numel, N: int, grad_bytes: int = 2, optim_bytes: int = 12) -> int:
    n = len(layer_numel)
    arr = (ctypes.c_int64 * max(n, 1))(*[int(x) for x in layer_numel])
    return _lib.zero3_peak_bytes(arr if n else None, n, N, grad_bytes, optim_bytes)


def zero_ledger(psi: int, N: int, stage: int, grad_bytes: int = 2, optim_bytes: int = 12) -> int:
    return _lib.zero_ledger(psi, N, stage, grad_bytes, optim_bytes)


def zero_comm_volume(psi: int, N: int, stage: int) -> int:
    return _lib.zero_comm_volume(psi, N, stage)


def zero_status_str(status: int) -> str:
    return _lib.zero_status_str(status).decode()


def zero_launch_count() -> int:
    return _lib.zero_launch_count()


def zero_debug_bounds_violations() -> int:
    """Out-of-range accesses the debug build's kernels skipped since the last
    call (and resets the count); -1 for the release build."""
    return _lib.zero_debug_bounds_violations()


def exported_symbols() -> list[str]:
    """Names of the C functions this binding expects the library to export."""
    return ["zero_init_layout", "zero_shard_range", "zero_workspace_bytes", "zero_step",
            "zero_step_into", "zero_plan_init", "zero_plan_init_ex",
            "zero_plan_set_device_policy", "zero_policy_table_fill",
            "zero_plan_set_device_policy_table", "zero_plan_set_pingpong", "zero_plan_begin",
            "zero_plan_bucket",
            "zero_plan_end", "zero_ledger", "zero_comm_volume", "zero_status_str",
            "zero_launch_count", "zero_step_noalloc", "zero3_gather", "zero3_peak_bytes",
            "zero_debug_bounds_violations"]
