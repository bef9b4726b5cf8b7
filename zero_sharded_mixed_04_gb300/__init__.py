"""GB300-native ZeRO sharded mixed-precision update step.

The step reduce-scatters N data-parallel ranks' gradients with batch-mean
scaling, applies mixed-precision Adam/AdamW on each owner's FP32
master/m/v slice, casts the updated master to BF16 and all-gathers it into
the full working-weight view.  The N ranks are simulated inside one GPU's
memory.  Every step runs in the hand-written CUDA kernels of
``libzero_gb300.so``.  The Python side only marshals arguments.

The C-ABI binding (``zero_step``, ``zero_init_layout``, ``zero_ledger``, ...)
lives in ``zero_sharded_mixed_04_gb300.zero``; it loads the shared library on
import and raises if that library has not been built, rather than falling back
to anything else.  Names not found here are looked up there on first use.
"""
from __future__ import annotations

import importlib

_SUBMODULES = ("zero", "synth", "build", "optim", "hostmem")


def __getattr__(name):
    if name.startswith("__"):
        raise AttributeError(name)
    if name in _SUBMODULES:
        return importlib.import_module(f"{__name__}.{name}")
    zero = importlib.import_module(f"{__name__}.zero")
    try:
        return getattr(zero, name)
    except AttributeError:
        raise AttributeError(f"module {__name__!r} has no attribute {name!r}") from None
