"""Every kernel writes only inside its buffers.

Each device buffer is carved from a larger allocation, with 4 KiB guard
regions filled with a pattern on both sides.  Steps of every form run, and
then the guards must be intact:
  - the one-pass, two-pass and out-of-place steps;
  - the one-pass step staged in shared memory by TMA, in and out of place;
  - clipping and accumulation;
  - the device policy;
  - the ZeRO-3 gather.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side


class Guarded:
    def __init__(self, numel, dtype, dev, fill=None):
        item = torch.empty((), dtype=dtype).element_size()
        g = GUARD // item
        self.base = torch.empty(numel + 2 * g, dtype=dtype, device=dev)
        self.base.view(torch.uint8).fill_(0xA5)
        self.g = g
        self.t = self.base[g:g + numel]
        if fill is not None:
            self.t.copy_(fill)

    def intact(self):
        raw = self.base.view(torch.uint8)
        gb = GUARD
        return bool((raw[:gb] == 0xA5).all() and (raw[-gb:] == 0xA5).all())


@pytest.mark.parametrize("form", ["one_pass", "two_pass_skip", "out_of_place_clip", "accumulate",
                                  "device_policy", "staged", "staged_out_of_place_skip"])
def test_guards_intact_after_steps(zero_lib, form):
    Z = zero_lib
    dev = torch.device("cuda:0")
    N, n = 4, 4 * 128 * 300 + 4 * 128 * 7
    gen = torch.Generator().manual_seed(4)
    k = 3 if form == "accumulate" else 1
    grads = [[Guarded(n, torch.bfloat16, dev, (torch.randn(n, generator=gen) * 1e-3).to(
        torch.bfloat16).to(dev)) for _ in range(N)] for _ in range(k)]
    src = [Guarded(n, torch.float32, dev, torch.randn(n, generator=gen).to(dev) * 0.02),
           Guarded(n, torch.float32, dev, torch.zeros(n, device=dev)),
           Guarded(n, torch.float32, dev, torch.zeros(n, device=dev)),
           Guarded(n, torch.int16, dev, torch.zeros(n, dtype=torch.int16, device=dev))]
    out_of_place = form in ("out_of_place_clip", "device_policy", "staged_out_of_place_skip")
    dst = [Guarded(n, x.t.dtype, dev, torch.zeros_like(x.t)) for x in src] if out_of_place else src
    hp = Z.make_hparams(skip_on_overflow=form in ("two_pass_skip", "device_policy",
                                                  "staged_out_of_place_skip"),
                        max_grad_norm=0.1 if form == "out_of_place_clip" else 0.0,
                        micro_batches=k, bucket_elems=4 * 128 * 64)
    ws_bytes = Z.zero_workspace_bytes(n, hp, not out_of_place)
    ws = Guarded(ws_bytes, torch.uint8, dev)
    res = Guarded(4, torch.int32, dev)
    plan = Z.zero_plan()
    assert Z.zero_plan_init(plan, [g.t for g in grads[0]], Z.ZERO_GRAD_BF16,
                            *[x.t for x in src], *[x.t for x in dst], n, N, hp, 1.0, ws.t,
                            ws_bytes) == Z.ZERO_OK
    plan.overlap_buckets = 1
    if form.startswith("staged"):
        plan.smem_staging = Z.ZERO_STAGING_TMA
    if form == "device_policy":
        pol_mem = torch.zeros(ctypes.sizeof(Z.zero_device_policy), dtype=torch.uint8,
                              pin_memory=True)
        pol = Z.zero_device_policy.from_address(pol_mem.data_ptr())
        pol.loss_scale = 1.0
        assert Z.zero_plan_set_device_policy(plan, pol_mem, 1, 1) == Z.ZERO_OK
    assert Z.zero_plan_begin(plan, None) == Z.ZERO_OK
    for mb in range(k):
        for b0 in range(0, n, 4 * 128 * 64):
            b1 = min(n, b0 + 4 * 128 * 64)
            assert Z.zero_plan_bucket(plan, b0, b1, [g.t[b0:b1] for g in grads[mb]],
                                      None) == Z.ZERO_OK
    assert Z.zero_plan_end(plan, res.t, None) == Z.ZERO_OK
    torch.cuda.synchronize()
    assert int(res.t[0].cpu()) == Z.ZERO_OK
    for x in [g for mb in grads for g in mb] + src + (dst if out_of_place else []) + [ws, res]:
        assert x.intact()


def test_guards_intact_after_gather(zero_lib):
    Z = zero_lib
    dev = torch.device("cuda:0")
    N, S = 4, 4096
    shards = [Guarded(S, torch.int16, dev, torch.arange(S, dtype=torch.int16, device=dev) + r)
              for r in range(N)]
    for b, e in [(0, N * S), (8, 8 + 3000), (5, 5 + 4091), (S - 3, S + 9)]:
        view = Guarded(e - b, torch.int16, dev, torch.zeros(e - b, dtype=torch.int16, device=dev))
        assert Z.zero3_gather([x.t for x in shards], N, S, b, e, view.t, None) == Z.ZERO_OK
        torch.cuda.synchronize()
        assert view.intact() and all(x.intact() for x in shards)
