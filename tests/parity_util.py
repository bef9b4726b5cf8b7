"""Shared helpers of the GPU parity tests: compare the CUDA path's state with
the oracle's, element by element, at the tolerances of the contract.

* Without clipping the two compute the same FP32 operators in the same order,
  so master/m/v and the BF16 weights must match bit for bit (a NaN matches
  any NaN).
* With clipping the norm is summed in a different order (a tree on the GPU,
  sequential in the oracle).  The FP32 clip coefficient may then differ in its
  last place, so master/m/v must agree within a relative 1e-6 and the BF16
  weights within 1 unit in the last place.
"""
from __future__ import annotations

import numpy as np

REL_TOL = 1e-6
BF16_ULP = 1


def _nan_aware_equal(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    if a.dtype == np.uint16:
        an = ((a & 0x7F80) == 0x7F80) & ((a & 0x7F) != 0)
        bn = ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)
        return (a == b) | (an & bn)
    return (a.view(np.uint32) == b.view(np.uint32)) | (np.isnan(a) & np.isnan(b))


def _first_bad(ok: np.ndarray) -> int:
    return int(np.flatnonzero(~ok)[0])


def assert_exact(name: str, got: np.ndarray, ref: np.ndarray, offset: int = 0) -> None:
    ok = _nan_aware_equal(got, ref)
    if not ok.all():
        i = _first_bad(ok)
        raise AssertionError(f"{name}: {int((~ok).sum())} elements differ; first at "
                             f"{offset + i}: got {got[i]!r} want {ref[i]!r}")


def assert_close(name: str, got: np.ndarray, ref: np.ndarray, offset: int = 0) -> None:
    if got.dtype == np.uint16:
        # BF16 within one unit in the last place: the integer distance of the
        # sign-magnitude bit patterns
        def key(h):
            h = h.astype(np.int32)
            return np.where(h & 0x8000, -(h & 0x7FFF), h)
        ok = (np.abs(key(got) - key(ref)) <= BF16_ULP) | _nan_aware_equal(got, ref)
    else:
        a, b = got.astype(np.float64), ref.astype(np.float64)
        ok = (np.abs(a - b) <= REL_TOL * np.abs(b) + 1e-30) | _nan_aware_equal(got, ref)
    if not ok.all():
        i = _first_bad(ok)
        raise AssertionError(f"{name}: {int((~ok).sum())} elements outside tolerance; first at "
                             f"{offset + i}: got {got[i]!r} want {ref[i]!r}")


def compare_state(gpu: dict, ref: dict, exact: bool, offset: int = 0, tag: str = "") -> None:
    check = assert_exact if exact else assert_close
    for k in ("master", "m", "v", "w"):
        check(f"{tag}{k}", gpu[k], ref[k], offset)


def compare_result(gpu: dict, ref: dict, exact_norm: bool = False) -> None:
    assert gpu["applied"] == ref["applied"], (gpu, ref)
    assert gpu["found_nonfinite"] == ref["found_nonfinite"], (gpu, ref)
    gn, rn = gpu["grad_norm"], ref["grad_norm"]
    if np.isfinite(rn):
        assert abs(gn - rn) <= REL_TOL * abs(rn), (gn, rn)
    else:
        assert not np.isfinite(gn), (gn, rn)
    assert abs(gpu["clip_coef"] - ref["clip_coef"]) <= REL_TOL * abs(ref["clip_coef"]) + 1e-30, \
        (gpu, ref)


def state_to_numpy(state: dict, lo: int = 0, hi: int | None = None) -> dict:
    """master/m/v (FP32) and w (BF16 bits) of a ZeroAdam state, on the host."""
    sl = slice(lo, hi)
    return {"master": state["master"][sl].cpu().numpy(), "m": state["m"][sl].cpu().numpy(),
            "v": state["v"][sl].cpu().numpy(),
            "w": state["w"][sl].cpu().numpy().view(np.uint16)}
