"""A step captured once as a CUDA graph and replayed step after step.

With a device policy whose bias corrections come from a table in device
memory, no launch of a step depends on t: t, the loss scale and (out of place)
the current ping-pong set live on the device.  So one captured step can be
replayed for every t the table covers.  Each replay here gets fresh gradients
in the captured buffers, two of them an injected +inf, and is compared with
the oracle bit for bit, through more replays than the 16-value window a
launch can carry.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from parity_util import compare_result, compare_state, state_to_numpy

pytestmark = pytest.mark.gpu

N = 4
PSI = 300_001
PSI_PAD = -(-PSI // (N * 128)) * (N * 128)


def _grads(seed: int, scale: float) -> list[torch.Tensor]:
    g = torch.Generator().manual_seed(seed)
    out = []
    for _ in range(N):
        z = torch.zeros(PSI_PAD)
        z[:PSI] = torch.randn(PSI, generator=g) * (1e-3 * scale)
        out.append(z.to(torch.bfloat16))
    return out


def _np(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).numpy().view(np.uint16)


def _optimizer(out_of_place: bool, staging: int, table_steps: int, master: torch.Tensor):
    from zero_sharded_mixed_04_gb300.optim import ZeroAdam
    return ZeroAdam(PSI_PAD, N, "bf16", lr=1e-3, weight_decay=0.01, skip_on_overflow=True,
                    bucket_elems=65_536, loss_scale=1024.0, dynamic_loss_scale=True,
                    growth_interval=4, out_of_place=out_of_place, pingpong=out_of_place,
                    device_policy=True, policy_table_steps=table_steps, smem_staging=staging,
                    device="cuda:0", master=master.to("cuda:0"))


@pytest.mark.parametrize("out_of_place,staging", [(True, 1), (True, 0), (False, 0)])
def test_graph_replays_match_the_oracle(zero_lib, oracle_mod, out_of_place, staging):
    master = torch.zeros(PSI_PAD)
    master[:PSI] = torch.randn(PSI, generator=torch.Generator().manual_seed(11)) * 0.02
    opt = _optimizer(out_of_place, staging, 40, master)
    bufs = [torch.zeros(PSI_PAD, dtype=torch.bfloat16, device="cuda:0") for _ in range(N)]
    graph = opt.capture_step(bufs)
    ref = {"master": master.numpy().copy(), "m": np.zeros(PSI_PAD, np.float32),
           "v": np.zeros(PSI_PAD, np.float32), "w": np.zeros(PSI_PAD, np.uint16)}
    hp = oracle_mod.Hparams(lr=1e-3, weight_decay=0.01)
    o_t, o_scale, o_good = 0, 1024.0, 0
    for step in range(1, 25):
        g = _grads(step, o_scale)
        if step in (5, 17):
            g[step % N][123] = float("inf")
        for b, x in zip(bufs, g):
            b.copy_(x)
        graph.replay()
        torch.cuda.synchronize()
        res = opt.last_result()
        ores = oracle_mod.zero_step([_np(x) for x in g], ref["master"], ref["m"], ref["v"],
                                    ref["w"], hp, o_t + 1, o_scale, True)
        tag = f"replay {step}: "
        try:
            compare_result(res, ores)
        except AssertionError as e:
            raise AssertionError(tag + str(e)) from None
        assert res["applied"] == (step not in (5, 17)), tag
        if ores["applied"]:
            o_t += 1
        o_scale, o_good = oracle_mod.loss_scale_update(o_scale, o_good, ores["found_nonfinite"],
                                                       4, 0.5, 2.0)
        assert int(opt.policy.t) == o_t and float(opt.policy.loss_scale) == o_scale, tag
        compare_state(state_to_numpy(opt.state()), ref, True, tag=tag)
    opt.finish_pending()
    assert opt.t == o_t == 22 and opt.scaler.scale == o_scale


def test_graph_replay_past_the_table_changes_nothing(zero_lib):
    Z = zero_lib
    master = torch.randn(PSI_PAD, generator=torch.Generator().manual_seed(3)) * 0.02
    opt = _optimizer(True, 1, 2, master)
    bufs = [x.to("cuda:0") for x in _grads(1, 1024.0)]
    graph = opt.capture_step(bufs)
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert int(opt.policy.t) == 2 and int(opt.result_t[0]) == Z.ZERO_OK
    before = {k: v.clone() for k, v in opt.state().items()}
    graph.replay()  # t' = 3: past the table
    torch.cuda.synchronize()
    assert int(opt.result_t[0]) == Z.ZERO_ERR_POLICY_WINDOW
    assert int(opt.policy.t) == 2 and int(opt.policy.last_status) == Z.ZERO_ERR_POLICY_WINDOW
    after = opt.state()
    for k in before:
        assert torch.equal(before[k], after[k]), k


def test_capture_needs_the_table(zero_lib):
    from zero_sharded_mixed_04_gb300.optim import ZeroAdam
    opt = ZeroAdam(PSI_PAD, N, "bf16", out_of_place=True, pingpong=True, device_policy=True,
                   skip_on_overflow=True, device="cuda:0")
    bufs = [torch.zeros(PSI_PAD, dtype=torch.bfloat16, device="cuda:0") for _ in range(N)]
    with pytest.raises(ValueError, match="policy_table_steps"):
        opt.capture_step(bufs)
    with pytest.raises(ValueError, match="device policy"):
        ZeroAdam(PSI_PAD, N, "bf16", policy_table_steps=8, device="cuda:0")
