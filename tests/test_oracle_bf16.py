"""Pin of the oracle's FP32 -> BF16 rounding against torch's CPU cast (a
library routine) over every one of the 2^32 FP32 bit patterns, and of the
widening against the bit-level definition."""
import numpy as np
import pytest
import torch

CHUNK = 1 << 24


def _torch_bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _is_nan_bf16(h: np.ndarray) -> np.ndarray:
    return ((h & 0x7F80) == 0x7F80) & ((h & 0x007F) != 0)


class _Checker:
    """Compares one chunk of consecutive FP32 bit patterns at a time, reusing
    its buffers."""

    def __init__(self, oracle_mod):
        self.oracle = oracle_mod
        self.base = np.arange(CHUNK, dtype=np.uint32)
        self.bits = np.empty(CHUNK, dtype=np.uint32)
        self.ours = np.empty(CHUNK, dtype=np.uint16)
        self.ref_t = torch.empty(CHUNK, dtype=torch.bfloat16)
        self.ref = self.ref_t.view(torch.int16).numpy().view(np.uint16)
        self.eq = np.empty(CHUNK, dtype=bool)

    def check(self, start: int):
        np.add(self.base, np.uint32(start), out=self.bits)
        x = self.bits.view(np.float32)
        self.oracle.f32_to_bf16(x, out=self.ours)
        self.ref_t.copy_(torch.from_numpy(x))
        np.equal(self.ours, self.ref, out=self.eq)
        if self.eq.all():
            return
        # only NaN inputs may differ, and then both sides must give a NaN
        bad = np.flatnonzero(~self.eq)
        nan_ok = np.isnan(x[bad]) & _is_nan_bf16(self.ours[bad]) & _is_nan_bf16(self.ref[bad])
        if not nan_ok.all():
            i = int(bad[np.flatnonzero(~nan_ok)[0]])
            raise AssertionError(f"bits 0x{int(self.bits[i]):08x}: oracle 0x{int(self.ours[i]):04x} "
                                 f"torch 0x{int(self.ref[i]):04x}")


def test_bf16_rne_every_fp32_pattern(oracle_mod):
    checker = _Checker(oracle_mod)
    for start in range(0, 1 << 32, CHUNK):
        checker.check(start)


def test_bf16_rne_hand_cases(oracle_mod):
    cases = {
        0x3F800000: 0x3F80,  # 1.0
        0x3F808000: 0x3F80,  # exactly half, even kept -> down
        0x3F818000: 0x3F82,  # exactly half, odd kept -> up
        0x3F808001: 0x3F81,  # above half -> up
        0x3F807FFF: 0x3F80,  # below half -> down
        0x7F7FFFFF: 0x7F80,  # largest FP32 rounds to +inf in BF16
        0x7F7F7FFF: 0x7F7F,  # stays the largest finite BF16
        0x80000000: 0x8000,  # -0
        0x00000001: 0x0000,  # smallest subnormal rounds to +0
        0x7F800000: 0x7F80,  # +inf
        0xFF800000: 0xFF80,  # -inf
    }
    x = np.array(list(cases), dtype=np.uint32).view(np.float32)
    got = oracle_mod.f32_to_bf16(x)
    assert [int(h) for h in got] == list(cases.values())


def test_bf16_widening_is_exact(oracle_mod):
    h = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    f = oracle_mod.bf16_to_f32(h)
    ref = torch.from_numpy(h.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    same = (f.view(np.uint32) == ref.view(np.uint32)) | (np.isnan(f) & np.isnan(ref))
    assert same.all()
    # round trip: BF16 -> FP32 -> BF16 is the identity for non-NaN patterns
    back = oracle_mod.f32_to_bf16(f)
    nan = np.isnan(f)
    assert (back[~nan] == h[~nan]).all()
