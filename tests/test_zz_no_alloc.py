"""zero_step_noalloc against zero_step, on the GPU, through the C ABI.

zero_step_noalloc serves callers that cannot allocate device memory
themselves.  For example, a program whose device memory belongs to another
allocator or pool, or a plugin that is handed only the tensors it works on.
It runs the in-place step with its workspace in a fixed array inside the
library.  This file checks that, for the same inputs, it gives what zero_step
with a caller-allocated workspace gives, and what the oracle gives.  The
check covers two calls in a row (the second reusing the array the first left
behind), that a call allocates no device memory, and the size limit of the
two-pass form.  Comparisons use the parity tests' tolerances: bit for bit
without clipping, within 1e-6 relative (BF16 within one unit in the last
place) with it.

The file name makes pytest collect it last.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from parity_util import compare_result, compare_state, state_to_numpy

pytestmark = pytest.mark.gpu


def _setup(N, psi, dtype, seed):
    dev = torch.device("cuda:0")
    unit = N * 128
    psi_pad = -(-psi // unit) * unit
    gen = torch.Generator().manual_seed(seed)
    master = torch.zeros(psi_pad)
    master[:psi] = torch.randn(psi, generator=gen) * 0.02
    sets = []
    for _ in range(2):
        sets.append({"master": master.to(dev),
                     "m": torch.zeros(psi_pad, device=dev), "v": torch.zeros(psi_pad, device=dev),
                     "w": torch.zeros(psi_pad, dtype=torch.int16, device=dev)})
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32

    def grads(step, bad=False):
        g = torch.Generator().manual_seed(seed * 100 + step)
        out = []
        for _ in range(N):
            z = torch.zeros(psi_pad)
            z[:psi] = torch.randn(psi, generator=g) * 1e-3 * 1024
            out.append(z.to(tdt).to(dev))
        if bad:
            out[N - 1][psi // 2] = float("inf")
        return out
    return psi_pad, sets, grads


def synth_np(t):
    """A device gradient buffer as the oracle takes it (a byte copy)."""
    from zero_sharded_mixed_04_gb300 import synth
    return synth.to_numpy_grad(t)


def _result(t):
    raw = t.cpu()
    return (int(raw[0]), int(raw[1]), float(raw[2:3].view(torch.float32)[0]),
            float(raw[3:4].view(torch.float32)[0]))


@pytest.mark.parametrize("N,psi,dtype,skip,clip,wd", [
    (4, 6_000_003, "bf16", False, 0.0, 0.1),   # one pass, larger than the two-pass limit
    (8, 3_000_017, "bf16", True, 0.0, 0.0),    # two passes (skip in place), overflow on call 2
    (4, 2_000_003, "fp32", False, 0.01, 0.0),  # two passes (clip)
])
def test_noalloc_matches_zero_step(zero_lib, oracle_mod, N, psi, dtype, skip, clip, wd):
    Z = zero_lib
    psi_pad, (a, b), grads = _setup(N, psi, dtype, seed=N + psi % 97)
    gdt = Z.ZERO_GRAD_BF16 if dtype == "bf16" else Z.ZERO_GRAD_FP32
    hp = Z.make_hparams(weight_decay=wd, max_grad_norm=clip, skip_on_overflow=skip)
    ws = torch.empty(Z.zero_workspace_bytes(psi_pad, hp, True), dtype=torch.uint8,
                     device="cuda:0")
    ra = torch.zeros(4, dtype=torch.int32, pin_memory=True)
    rb = torch.zeros(4, dtype=torch.int32, pin_memory=True)
    ref = state_to_numpy(a)
    ohp = oracle_mod.Hparams(weight_decay=wd, max_grad_norm=clip)
    t = 0
    for call in (1, 2):
        g = grads(call, bad=skip and call == 2)
        hp.step = t + 1
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        reserved_before = torch.cuda.memory_reserved()
        rc = Z.zero_step_noalloc(g, gdt, a["master"], a["m"], a["v"], a["w"], psi_pad, N, hp,
                                 1024.0, ra, None)
        assert rc == Z.ZERO_OK, Z.zero_status_str(rc)
        torch.cuda.synchronize()
        if call == 2:
            # the first call may load the library's device code (and with it
            # the fixed array); a later call allocates nothing at all
            assert torch.cuda.mem_get_info()[0] == free_before
            assert torch.cuda.memory_reserved() == reserved_before
        rc = Z.zero_step(g, gdt, b["master"], b["m"], b["v"], b["w"], psi_pad, N, hp, 1024.0,
                         ws, ws.numel(), rb, None)
        assert rc == Z.ZERO_OK, Z.zero_status_str(rc)
        torch.cuda.synchronize()
        res_a, res_b = _result(ra), _result(rb)
        assert res_a[:2] == res_b[:2]
        assert res_a[0] == (Z.ZERO_STEP_SKIPPED if skip and call == 2 else Z.ZERO_OK)
        np.testing.assert_allclose(res_a[2:], res_b[2:], rtol=1e-6)
        compare_state(state_to_numpy(a), state_to_numpy(b), exact=clip == 0.0,
                      tag=f"call {call} ")
        # and the oracle on the same gradients
        ores = oracle_mod.zero_step([synth_np(x) for x in g], ref["master"], ref["m"], ref["v"],
                                    ref["w"], ohp, t + 1, 1024.0, skip)
        compare_result({"applied": res_a[0] == Z.ZERO_OK, "found_nonfinite": bool(res_a[1]),
                        "grad_norm": res_a[2], "clip_coef": res_a[3]}, ores)
        compare_state(state_to_numpy(a), ref, exact=clip == 0.0, tag=f"oracle, call {call} ")
        if res_a[0] == Z.ZERO_OK:
            t += 1


def test_noalloc_rejects_two_pass_beyond_its_array(zero_lib):
    Z = zero_lib
    N = 4
    psi_pad = Z.ZERO_NOALLOC_MAX_TWO_PASS_ELEMS + N * 128
    dev = torch.device("cuda:0")
    st = [torch.zeros(psi_pad, device=dev) for _ in range(3)]
    w = torch.zeros(psi_pad, dtype=torch.int16, device=dev)
    g = [torch.zeros(psi_pad, dtype=torch.bfloat16, device=dev) for _ in range(N)]
    for hp in (Z.make_hparams(skip_on_overflow=True), Z.make_hparams(max_grad_norm=1.0)):
        rc = Z.zero_step_noalloc(g, Z.ZERO_GRAD_BF16, *st, w, psi_pad, N, hp, 1.0, None, None)
        assert rc == Z.ZERO_ERR_TOO_LARGE
        assert "scratch" in Z.zero_status_str(rc)
    # nothing was touched
    assert not st[0].any() and not w.any()
    # at the limit the two-pass form is accepted
    at = Z.ZERO_NOALLOC_MAX_TWO_PASS_ELEMS
    rc = Z.zero_step_noalloc([x[:at] for x in g], Z.ZERO_GRAD_BF16, st[0][:at], st[1][:at],
                             st[2][:at], w[:at], at, N, Z.make_hparams(skip_on_overflow=True),
                             1.0, None, None)
    assert rc == Z.ZERO_OK
