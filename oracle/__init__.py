"""CPU oracle for the ZeRO sharded mixed-precision update step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product library
(``zero_sharded_mixed_04_gb300``) never does, and this package imports nothing
from it.

The arithmetic lives in ``zero_oracle.c`` (plain C, FP32 operators rounded one
at a time, compiled without FMA contraction or fast-math).  This module only
compiles it with gcc on first use and marshals numpy arrays through ctypes.

Pins (what ties this oracle to something other than itself) are in
``tests/test_oracle_*.py``: the pages' printed ledger numbers, the
reduce-scatter/all-gather = all-reduce identity, the ZeRO step = the DDP step,
torch's CPU AdamW / BF16 cast / gradient clipping / loss-scale update as
library special cases, closed forms of Adam's first steps and brute force on
integer-valued tiny cases.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zero_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libzero_oracle.so")
# the same source built with OpenMP: the all-cores timing mode (CPU baseline only)
_LIB_OMP_PATH = os.path.join(_HERE, "libzero_oracle_omp.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

BF16 = 0
FP32 = 1
PAD_UNIT = 128

_lock = threading.Lock()
_lib = None
_lib_omp = None


def build(force: bool = False, parallel: bool = False) -> str:
    """Compile the oracle's C source into a shared library next to it
    (``parallel``: the OpenMP build of the same source)."""
    path = _LIB_OMP_PATH if parallel else _LIB_PATH
    stale = not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = path + f".tmp{os.getpid()}"
        extra = ["-fopenmp"] if parallel else []
        subprocess.run(["gcc", *_CFLAGS, *extra, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, path)
    return path


class _Hparams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_double) for n in
                ("lr", "beta1", "beta2", "eps", "weight_decay", "max_grad_norm")]


class _Scalars(ctypes.Structure):
    _fields_ = [("inv", ctypes.c_float), ("b1", ctypes.c_float), ("omb1", ctypes.c_float),
                ("b2", ctypes.c_float), ("omb2", ctypes.c_float), ("eps", ctypes.c_float),
                ("step_size", ctypes.c_float), ("sbc2", ctypes.c_float),
                ("decay", ctypes.c_float), ("use_decay", ctypes.c_int32)]


class _Result(ctypes.Structure):
    _fields_ = [("applied", ctypes.c_int32), ("found_nonfinite", ctypes.c_int32),
                ("sumsq", ctypes.c_double), ("grad_norm", ctypes.c_float),
                ("clip_coef", ctypes.c_float)]


def _declare(lib):
    P = ctypes.c_void_p
    i32, i64, f32, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_double
    lib.orc_f32_to_bf16_array.argtypes = [P, P, i64]
    lib.orc_f32_to_bf16.argtypes = [f32]
    lib.orc_f32_to_bf16.restype = ctypes.c_uint16
    lib.orc_layout.argtypes = [P, i64, i32, P, P, P, P]
    lib.orc_layout.restype = i32
    lib.orc_ledger_bytes.argtypes = [i64, i32, i32, i32, i32]
    lib.orc_ledger_bytes.restype = i64
    lib.orc_comm_volume.argtypes = [i64, i32, i32, i32]
    lib.orc_comm_volume.restype = i64
    lib.orc_step_scalars.argtypes = [P, i64, i32, f64, P]
    lib.orc_reduce_scatter.argtypes = [P, i32, i32, i64, i32, f32, P]
    lib.orc_all_reduce.argtypes = [P, i32, i32, i64, f32, P]
    lib.orc_all_gather_f32.argtypes = [P, i32, i64, P]
    lib.orc_zero_step.argtypes = [P, i32, i32, i64, P, P, P, P, P, i64, f64, i32, P]
    lib.orc_zero_step.restype = i32
    lib.orc_ddp_step.argtypes = [P, i32, i32, i64, P, P, P, P, P, i64, f64, i32, P]
    lib.orc_ddp_step.restype = i32
    lib.orc_zero_step_accum.argtypes = [P, i32, i32, i32, i64, P, P, P, P, P, i64, f64,
                                         i32, P]
    lib.orc_zero_step_accum.restype = i32
    lib.orc_gather_range.argtypes = [P, i32, i64, i64, i64, P]
    lib.orc_gather_range.restype = i32
    lib.orc_zero3_peak_bytes.argtypes = [P, i64, i32, i32, i32]
    lib.orc_zero3_peak_bytes.restype = i64
    lib.orc_check_accumulate.argtypes = [P, i32, i32, i64, f32, P, P]
    lib.orc_step_window.argtypes = [P, i32, i32, i64, P, P, P, P, P, i64, f64,
                                    i32, i32, f32]
    lib.orc_clip_coef_from_sumsq.argtypes = [f64, f64]
    lib.orc_clip_coef_from_sumsq.restype = f32
    lib.orc_loss_scale_update.argtypes = [P, P, i32, i32, f64, f64]
    return lib


def _load(parallel: bool = False):
    global _lib, _lib_omp
    with _lock:
        if parallel:
            if _lib_omp is None:
                _lib_omp = _declare(ctypes.CDLL(build(parallel=True)))
            return _lib_omp
        if _lib is None:
            # ORACLE_LIB_OVERRIDE loads another build of the oracle's source;
            # only the mutation test uses it, to check that the pins catch
            # planted mistakes
            override = os.environ.get("ORACLE_LIB_OVERRIDE")
            _lib = _declare(ctypes.CDLL(override if override else build()))
    return _lib


@dataclass
class Hparams:
    """Adam/AdamW hyper-parameters (FP64, as a host would hold them)."""
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    max_grad_norm: float = 0.0  # 0 = no clipping

    def _c(self) -> _Hparams:
        return _Hparams(self.lr, self.beta1, self.beta2, self.eps, self.weight_decay,
                        self.max_grad_norm)


def _ptr(a: np.ndarray) -> int:
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("oracle arrays must be C-contiguous")
    return a.ctypes.data


def _grad_dtype(grads) -> int:
    dt = grads[0].dtype
    if any(g.dtype != dt for g in grads):
        raise ValueError("all ranks' gradients must share one dtype")
    if dt == np.uint16:
        return BF16
    if dt == np.float32:
        return FP32
    raise ValueError("gradients are BF16 bit patterns (uint16) or float32")


def _ptr_array(arrays):
    return (ctypes.c_void_p * len(arrays))(*[_ptr(a) for a in arrays])


# --------------------------------------------------------------------------- scalars

def f32_to_bf16(x: np.ndarray, out: np.ndarray | None = None) -> np.ndarray:
    """Round-to-nearest-even FP32 -> BF16 bit patterns (uint16)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if out is None:
        out = np.empty(x.shape, dtype=np.uint16)
    _load().orc_f32_to_bf16_array(_ptr(x), _ptr(out), x.size)
    return out


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    """Exact widening of BF16 bit patterns to FP32."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def layout(numel, N: int):
    """(offsets, psi, psi_pad, shard) of the flat, padded, sharded vector."""
    numel = np.ascontiguousarray(numel, dtype=np.int64)
    offsets = np.empty(max(numel.size, 1), dtype=np.int64)
    psi, psi_pad, shard = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    rc = _load().orc_layout(_ptr(numel) if numel.size else None, numel.size, N,
                            _ptr(offsets), ctypes.byref(psi), ctypes.byref(psi_pad),
                            ctypes.byref(shard))
    if rc != 0:
        raise ValueError("bad layout arguments")
    return offsets[:numel.size], psi.value, psi_pad.value, shard.value


def ledger_bytes(psi: int, N: int, stage: int, grad_bytes: int = 2, optim_bytes: int = 12) -> int:
    return _load().orc_ledger_bytes(psi, N, stage, grad_bytes, optim_bytes)


def comm_volume(psi: int, N: int, stage: int, ring_exact: bool = False) -> int:
    return _load().orc_comm_volume(psi, N, stage, int(ring_exact))


def step_scalars(hp: Hparams, t: int, N: int, loss_scale: float) -> dict:
    s = _Scalars()
    c = hp._c()
    _load().orc_step_scalars(ctypes.byref(c), t, N, loss_scale, ctypes.byref(s))
    return {name: getattr(s, name) for name, _ in _Scalars._fields_}


def clip_coef_from_sumsq(max_norm: float, sumsq: float) -> float:
    return _load().orc_clip_coef_from_sumsq(max_norm, sumsq)


def loss_scale_update(scale: float, good_steps: int, found_nonfinite: bool,
                      interval: int = 2000, backoff: float = 0.5, growth: float = 2.0):
    """Dynamic loss-scale policy; returns (new_scale, new_good_steps)."""
    s = ctypes.c_double(scale)
    g = ctypes.c_int32(good_steps)
    _load().orc_loss_scale_update(ctypes.byref(s), ctypes.byref(g), int(bool(found_nonfinite)),
                                  interval, backoff, growth)
    return s.value, g.value


def gather_range(shards, begin: int, end: int) -> np.ndarray:
    """Elements [begin, end) of the full view, from N BF16 shards (uint16)."""
    shards = [np.ascontiguousarray(x, dtype=np.uint16) for x in shards]
    out = np.empty(max(end - begin, 1), dtype=np.uint16)
    rc = _load().orc_gather_range(_ptr_array(shards), len(shards), shards[0].size, begin, end,
                                  _ptr(out))
    if rc != 0:
        raise ValueError("bad gather range")
    return out[:end - begin]


def zero3_peak_bytes(layer_numel, N: int, grad_bytes: int = 2, optim_bytes: int = 12) -> int:
    """Peak bytes per rank under ZeRO-3 with the two-view gather schedule."""
    arr = np.ascontiguousarray(layer_numel, dtype=np.int64)
    return _load().orc_zero3_peak_bytes(_ptr(arr) if arr.size else None, arr.size, N, grad_bytes,
                                        optim_bytes)


# --------------------------------------------------------------------------- collectives

def reduce_scatter(grads, psi_pad: int, r: int, inv: float) -> np.ndarray:
    N = len(grads)
    out = np.empty(psi_pad // N, dtype=np.float32)
    _load().orc_reduce_scatter(_ptr_array(grads), _grad_dtype(grads), N, psi_pad, r, inv,
                               _ptr(out))
    return out


def all_reduce(grads, psi_pad: int, inv: float) -> np.ndarray:
    N = len(grads)
    out = np.empty(psi_pad, dtype=np.float32)
    _load().orc_all_reduce(_ptr_array(grads), _grad_dtype(grads), N, psi_pad, inv, _ptr(out))
    return out


def all_gather_f32(shards) -> np.ndarray:
    shards = [np.ascontiguousarray(s, dtype=np.float32) for s in shards]
    shard = shards[0].size
    out = np.empty(shard * len(shards), dtype=np.float32)
    _load().orc_all_gather_f32(_ptr_array(shards), len(shards), shard, _ptr(out))
    return out


# --------------------------------------------------------------------------- the step

def _result(r: _Result) -> dict:
    return {"applied": bool(r.applied), "found_nonfinite": bool(r.found_nonfinite),
            "sumsq": r.sumsq, "grad_norm": r.grad_norm, "clip_coef": r.clip_coef}


def zero_step(grads, master, m, v, w, hp: Hparams, t: int, loss_scale: float = 1.0,
              skip_on_overflow: bool = False, parallel: bool = False) -> dict:
    """One ZeRO step (owner form) in place on flat master/m/v (float32) and w
    (BF16 bits, uint16), all of psi_pad elements; grads is a list of N arrays.
    ``parallel`` runs the OpenMP build (the CPU baseline's all-cores mode):
    the same elements, the norm in fixed-order per-thread partials."""
    N = len(grads)
    res = _Result()
    c = hp._c()
    rc = _load(parallel).orc_zero_step(_ptr_array(grads), _grad_dtype(grads), N, master.size,
                               _ptr(master), _ptr(m), _ptr(v), _ptr(w), ctypes.byref(c), t,
                               loss_scale, int(skip_on_overflow), ctypes.byref(res))
    if rc != 0:
        raise ValueError("oracle zero_step rejected its arguments")
    return _result(res)


def zero_step_accum(micro_grads, master, m, v, w, hp: Hparams, t: int, loss_scale: float = 1.0,
                    skip_on_overflow: bool = False) -> dict:
    """One step on the gradient accumulated over k micro-batches.
    micro_grads[mb] is the list of N ranks' gradients of micro-batch mb."""
    k = len(micro_grads)
    N = len(micro_grads[0])
    flat = [g for mb in micro_grads for g in mb]
    res = _Result()
    c = hp._c()
    rc = _load().orc_zero_step_accum(_ptr_array(flat), _grad_dtype(flat), N, k, master.size,
                                     _ptr(master), _ptr(m), _ptr(v), _ptr(w), ctypes.byref(c), t,
                                     loss_scale, int(skip_on_overflow), ctypes.byref(res))
    if rc != 0:
        raise ValueError("oracle zero_step_accum rejected its arguments")
    return _result(res)


def ddp_step(grads, masters, ms, vs, ws, hp: Hparams, t: int, loss_scale: float = 1.0,
             skip_on_overflow: bool = False) -> dict:
    """One replicated (DDP) step: replica i updates masters[i], ms[i], vs[i], ws[i]."""
    N = len(grads)
    res = _Result()
    c = hp._c()
    rc = _load().orc_ddp_step(_ptr_array(grads), _grad_dtype(grads), N, masters[0].size,
                              _ptr_array(masters), _ptr_array(ms), _ptr_array(vs),
                              _ptr_array(ws), ctypes.byref(c), t, loss_scale,
                              int(skip_on_overflow), ctypes.byref(res))
    if rc != 0:
        raise ValueError("oracle ddp_step rejected its arguments")
    return _result(res)


class CheckAccumulator:
    """Step-wide overflow flag and FP64 sum of squares, fed chunk by chunk in
    flat order (the same sequential sum the whole-vector step takes)."""

    def __init__(self, N: int, loss_scale: float = 1.0):
        self.N = N
        self.inv = np.float32(1.0 / (N * loss_scale))
        self._bad = ctypes.c_int32(0)
        self._sumsq = ctypes.c_double(0.0)

    def feed(self, grads_chunk) -> None:
        if len(grads_chunk) != self.N:
            raise ValueError("one chunk per rank")
        _load().orc_check_accumulate(_ptr_array(grads_chunk), _grad_dtype(grads_chunk), self.N,
                                     grads_chunk[0].size, float(self.inv),
                                     ctypes.byref(self._bad), ctypes.byref(self._sumsq))

    @property
    def found_nonfinite(self) -> bool:
        return bool(self._bad.value)

    @property
    def sumsq(self) -> float:
        return self._sumsq.value


def step_window(grads_window, master, m, v, w, hp: Hparams, t: int, loss_scale: float,
                apply: bool, clip_coef: float | None) -> None:
    """Step a window of the flat vector in place, given the step-wide outcome."""
    N = len(grads_window)
    c = hp._c()
    _load().orc_step_window(_ptr_array(grads_window), _grad_dtype(grads_window), N, master.size,
                            _ptr(master), _ptr(m), _ptr(v), _ptr(w), ctypes.byref(c), t,
                            loss_scale, int(apply), int(clip_coef is not None),
                            1.0 if clip_coef is None else clip_coef)
