"""Shared helpers of the GPU parity tests: compare the CUDA path's state with
the oracle's, element by element, at the tolerances of the contract.

* Without clipping the two compute the same FP32 operators in the same order,
  so master/m/v and the BF16 weights must match bit for bit (a NaN matches
  any NaN).
* With clipping the norm is summed in a different order (a tree on the GPU,
  sequential in the oracle).  The FP32 clip coefficient may then differ in its
  last place, so master/m/v must agree within a relative 1e-6 and the BF16
  weights within 1 unit in the last place.  "Relative" is taken against the
  larger of the element and the array's RMS: an element formed by
  cancellation (p - step close to 0, or beta1*m + (1-beta1)*g close to 0)
  carries the rounding of its operands, whose size is the array's, not its
  own.  A weight is the master rounded to BF16, so it may also lie anywhere
  between the roundings of its master's tolerance interval (one unit
  further either way).
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


def _bf16_key(h: np.ndarray) -> np.ndarray:
    """BF16 bit patterns as integers ordered like their values (sign-magnitude)."""
    h = h.astype(np.int32)
    return np.where(h & 0x8000, -(h & 0x7FFF), h)


def _bf16_rne(x: np.ndarray) -> np.ndarray:
    """FP32 values rounded to BF16 bit patterns, nearest with ties to even."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def _fp32_tolerance(ref: np.ndarray) -> np.ndarray:
    """1e-6 relative to the larger of the element and the array's RMS."""
    b = ref.astype(np.float64)
    finite = b[np.isfinite(b)]
    rms = float(np.sqrt(np.mean(finite * finite))) if finite.size else 0.0
    return REL_TOL * np.abs(b) + REL_TOL * rms + 1e-30


def assert_close(name: str, got: np.ndarray, ref: np.ndarray, offset: int = 0,
                 master_ref: np.ndarray | None = None) -> None:
    if got.dtype == np.uint16:
        # BF16 within one unit in the last place: the integer distance of the
        # sign-magnitude bit patterns
        ok = (np.abs(_bf16_key(got) - _bf16_key(ref)) <= BF16_ULP) | _nan_aware_equal(got, ref)
        if master_ref is not None and not ok.all():
            # The weights are the master rounded to BF16.  Where they are
            # (ref equal to the rounded ref master), a master anywhere within
            # its tolerance may round to anything between the roundings of
            # the interval's ends, one unit further either way.
            tol = _fp32_tolerance(master_ref)
            mr = master_ref.astype(np.float64)
            lo = _bf16_key(_bf16_rne((mr - tol).astype(np.float32))) - BF16_ULP
            hi = _bf16_key(_bf16_rne((mr + tol).astype(np.float32))) + BF16_ULP
            cast = _bf16_rne(master_ref) == ref
            k = _bf16_key(got)
            ok |= cast & (k >= lo) & (k <= hi)
    else:
        a = got.astype(np.float64)
        ok = (np.abs(a - ref.astype(np.float64)) <= _fp32_tolerance(ref)) | _nan_aware_equal(got, ref)
    if not ok.all():
        i = _first_bad(ok)
        raise AssertionError(f"{name}: {int((~ok).sum())} elements outside tolerance; first at "
                             f"{offset + i}: got {got[i]!r} want {ref[i]!r}")


def compare_state(gpu: dict, ref: dict, exact: bool, offset: int = 0, tag: str = "") -> None:
    for k in ("master", "m", "v", "w"):
        if exact:
            assert_exact(f"{tag}{k}", gpu[k], ref[k], offset)
        else:
            assert_close(f"{tag}{k}", gpu[k], ref[k], offset,
                         master_ref=ref["master"] if k == "w" else None)


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
