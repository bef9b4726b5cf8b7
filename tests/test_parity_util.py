"""The GPU parity tests' comparison helpers, checked on the host."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import parity_util as pu


def test_bf16_rounding_matches_torch():
    g = torch.Generator().manual_seed(3)
    x = torch.randn(200_000, generator=g) * torch.logspace(-38, 38, 200_000)
    x[:6] = torch.tensor([0.0, -0.0, 1.0, float("inf"), -float("inf"), 3.0e38])
    want = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(pu._bf16_rne(x.numpy()), want)


def test_fp32_tolerance_has_a_floor_at_the_array_scale():
    ref = np.full(1000, 0.02, np.float32)
    ref[0] = -4.0016894e-05                        # formed by cancellation
    got = ref.copy()
    got[0] = np.float32(-4.0016836e-05)            # 5.8e-11 off: inside 1e-6 * rms
    pu.assert_close("master", got, ref)
    got[1] = np.float32(0.02 * (1 + 3e-6))         # 3e-6 relative at full size: outside
    with pytest.raises(AssertionError, match="1 elements outside"):
        pu.assert_close("master", got, ref)


def test_bf16_weights_follow_their_master_interval():
    master = np.full(1000, 0.02, np.float32)
    master[0] = 2.8e-8                             # a master formed by cancellation
    w = pu._bf16_rne(master)
    got = w.copy()
    got[0] = w[0] + 7                              # 2.9e-8: within 1e-6 * rms of 2.8e-8
    pu.assert_close("w", got, w, master_ref=master)
    got[5] = w[5] + 2                              # two units at full size: outside
    with pytest.raises(AssertionError):
        pu.assert_close("w", got, w, master_ref=master)
    # a weight that is not its master's rounding (a skipped first step) keeps the 1-unit rule
    stale = np.zeros(1000, np.uint16)
    got = stale.copy()
    got[0] = 7
    with pytest.raises(AssertionError):
        pu.assert_close("w", got, stale, master_ref=master)


def test_exact_comparison_is_unchanged():
    ref = {"master": np.array([1.0, np.nan], np.float32), "m": np.zeros(2, np.float32),
           "v": np.zeros(2, np.float32), "w": np.array([0x3F80, 0x7FC0], np.uint16)}
    got = {k: v.copy() for k, v in ref.items()}
    pu.compare_state(got, ref, exact=True)
    got["master"][0] = np.nextafter(np.float32(1.0), np.float32(2.0))
    with pytest.raises(AssertionError, match="differ"):
        pu.compare_state(got, ref, exact=True)
