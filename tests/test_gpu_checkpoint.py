"""Checkpoint and resume: k steps equal j steps, a save to the host, a load
into a fresh optimizer and k - j more steps, bit for bit (state, t and the
loss scale).  With and without the device-resident policy, in and out of
place (out of place also with ping-pong state sets, where the device keeps
which set is current), with an overflowing step before the checkpoint."""
from __future__ import annotations

import pytest
import torch

pytestmark = pytest.mark.gpu


def _grads(N, n, step, scale):
    g = torch.Generator().manual_seed(1000 + step)
    out = [(torch.randn(n, generator=g) * 1e-3 * scale).to(torch.bfloat16) for _ in range(N)]
    if step == 2:
        out[0][99] = float("inf")
    return out


@pytest.mark.parametrize("out_of_place,pingpong", [(False, False), (True, False), (True, True)])
@pytest.mark.parametrize("device_policy", [False, True])
def test_resume_is_bit_exact(out_of_place, pingpong, device_policy):
    from zero_sharded_mixed_04_gb300.optim import ZeroAdam
    dev = torch.device("cuda:0")
    N, n = 4, 4 * 128 * 500
    master = torch.randn(n, generator=torch.Generator().manual_seed(2)) * 0.02

    def make():
        return ZeroAdam(n, N, "bf16", weight_decay=0.1, skip_on_overflow=True, loss_scale=1024.0,
                        dynamic_loss_scale=True, growth_interval=2, out_of_place=out_of_place,
                        device=dev, master=master.to(dev), device_policy=device_policy,
                        pingpong=pingpong)

    def run(opt, steps):
        for s in steps:
            opt.step_async([g.to(dev) for g in _grads(N, n, s, opt.scaler.scale)])
            if device_policy:
                opt.finish_pending()   # the next step's gradients use the current scale

    a = make()
    run(a, range(1, 6))
    a.finish_pending()
    b = make()
    run(b, range(1, 3))
    sd = b.state_dict()
    c = make()
    c.load_state_dict(sd)
    run(c, range(3, 6))
    c.finish_pending()
    assert (c.t, c.scaler.scale, c.scaler.good_steps) == (a.t, a.scaler.scale, a.scaler.good_steps)
    assert a.t == 4  # step 2 overflowed
    for k in ("master", "m", "v", "w"):
        assert torch.equal(a.state()[k], c.state()[k]), k
    if pingpong:
        # a ran 4 applied steps from set 0; c restarted from set 0 after 1
        # applied step and applied 3 more: each ends on the set its count says
        assert int(a.set_mem[0]) == 0 and int(c.set_mem[0]) == 1
