"""GPU parity over a seeded random sweep of whole configurations.

The parity matrix of test_gpu_parity.py walks each option on its own.  Here
every case draws all of them at once from its own seed, so that options meet
in combinations no hand-written case lists:
  - N from 1 to 16, BF16 or FP32 gradients, a ragged size from 1 element up
    (one case in sixteen past the 2^22 elements of one launch);
  - lr, the betas, eps and weight decay;
  - clip (none, active, or a bound so large that it never bites);
  - skip on overflow, in place or out of place, ping-pong state sets;
  - t and the loss scale on the host or on the device, a static or dynamic
    loss scale;
  - one bucket or many, the zero_step or plan entry points, the register or
    the TMA-staged kernel;
  - one batch or 2-3 accumulated micro-batches;
  - a +inf, -inf or NaN planted in some step, micro-batch, rank and element;
  - eager steps, or one step captured as a CUDA graph and replayed.
Each case runs three steps through ZeroAdam (the library's public Python API)
and compares every step's outcome and state with the oracle: bit for bit
without clip, within the clip tolerance with it.  A failing case names its
seed, and draw_case(seed) rebuilds it.
"""
from __future__ import annotations

import random

import numpy as np
import pytest
import torch

from parity_util import compare_result, compare_state, state_to_numpy

pytestmark = pytest.mark.gpu

N_CASES = 256
STEPS = 3


def draw_case(seed: int) -> dict:
    r = random.Random(seed)
    long = r.random() < 1 / 16   # past one launch's 2^22 elements: a chain of sub-launches
    N = r.choice([1, 2, 3, 4]) if long else r.choice([1, 2, 3, 4, 5, 6, 7, 8, 9, 11, 16])
    dtype = r.choice(["bf16", "fp32"])
    psi = (r.randrange(4_200_000, 9_000_000) if long else
           r.choice([1, 7, 129, 1000, r.randrange(1, 50_000), r.randrange(50_000, 600_000),
                     r.randrange(600_000, 3_000_000)]))
    psi_pad = -(-psi // (N * 128)) * (N * 128)
    k = 1 if long else r.choice([1, 1, 1, 2, 3])
    out_of_place = r.random() < 0.5
    pingpong = out_of_place and r.random() < 0.5
    skip = r.random() < 0.5
    dynamic = r.random() < 0.4
    device_policy = (skip or dynamic) and r.random() < 0.4
    bucket = 0 if r.random() < 0.4 else 8 * r.randrange(8, max(9, psi_pad // 8 + 1))
    # the staged kernel holds two tiles of every rank in shared memory
    staging = int(r.random() < 0.5 and N <= (18 if dtype == "bf16" else 9))
    bad = None
    if r.random() < 0.35:
        bad = {"step": r.randrange(1, STEPS + 1), "micro": r.randrange(k), "rank": r.randrange(N),
               "index": r.randrange(psi), "value": r.choice([float("inf"), float("-inf"),
                                                              float("nan")])}
    return {
        "seed": seed, "N": N, "dtype": dtype, "psi": psi, "psi_pad": psi_pad, "k": k,
        "lr": r.choice([1e-3, 3e-4, 1e-2]), "beta1": r.choice([0.9, 0.8]),
        "beta2": r.choice([0.999, 0.95]), "eps": r.choice([1e-8, 1e-6]),
        "wd": r.choice([0.0, 0.0, 0.01, 0.1]), "clip": r.choice([0.0, 0.0, 0.0, 0.02, 1.0, 1e6]),
        "skip": skip, "out_of_place": out_of_place, "pingpong": pingpong, "dynamic": dynamic,
        "device_policy": device_policy, "bucket": bucket, "staging": staging,
        "api": "plan" if (staging or k > 1 or device_policy or pingpong)
        else r.choice(["step", "plan"]),
        "loss_scale": r.choice([1.0, 128.0, 4096.0]), "sigma": r.choice([1e-4, 1e-3, 3e-2]),
        "bad": bad,
        # drawn last, so that the other options of every seed stay as they were:
        # the step captured once as a CUDA graph and replayed (device policy
        # with a table of bias corrections; in place or with ping-pong sets)
        "graph": (device_policy and k == 1 and (pingpong or not out_of_place)
                  and r.random() < 0.5),
    }


def _grads(case, step, micro, scale):
    g = torch.Generator().manual_seed(case["seed"] * 1000 + step * 10 + micro)
    out = []
    for _ in range(case["N"]):
        z = torch.zeros(case["psi_pad"], dtype=torch.float32)
        z[:case["psi"]] = torch.randn(case["psi"], generator=g) * (case["sigma"] * scale)
        out.append(z.to(torch.bfloat16) if case["dtype"] == "bf16" else z)
    return out


def _np(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def run_case(case: dict, oracle_mod) -> None:
    """The case's three steps through ZeroAdam, each checked against the oracle."""
    from zero_sharded_mixed_04_gb300.optim import ZeroAdam
    seed = case["seed"]
    dev = torch.device("cuda:0")
    psi, psi_pad = case["psi"], case["psi_pad"]
    master = torch.zeros(psi_pad)
    master[:psi] = torch.randn(psi, generator=torch.Generator().manual_seed(seed + 17)) * 0.02
    opt = ZeroAdam(psi_pad, case["N"], case["dtype"], lr=case["lr"], beta1=case["beta1"],
                   beta2=case["beta2"], eps=case["eps"], weight_decay=case["wd"],
                   max_grad_norm=case["clip"], skip_on_overflow=case["skip"],
                   bucket_elems=case["bucket"], loss_scale=case["loss_scale"],
                   dynamic_loss_scale=case["dynamic"], growth_interval=2,
                   out_of_place=case["out_of_place"], device=dev, master=master.to(dev),
                   micro_batches=case["k"] if case["k"] > 1 else 0,
                   device_policy=case["device_policy"], smem_staging=case["staging"],
                   pingpong=case["pingpong"],
                   policy_table_steps=STEPS + 4 if case.get("graph") else 0)
    graph, bufs = None, None
    if case.get("graph"):
        tdt = torch.bfloat16 if case["dtype"] == "bf16" else torch.float32
        bufs = [torch.zeros(psi_pad, dtype=tdt, device=dev) for _ in range(case["N"])]
        graph = opt.capture_step(bufs)
    ref = {"master": master.numpy().copy(), "m": np.zeros(psi_pad, np.float32),
           "v": np.zeros(psi_pad, np.float32), "w": np.zeros(psi_pad, np.uint16)}
    hp = oracle_mod.Hparams(lr=case["lr"], beta1=case["beta1"], beta2=case["beta2"],
                            eps=case["eps"], weight_decay=case["wd"], max_grad_norm=case["clip"])
    o_t, o_scale, o_good = 0, case["loss_scale"], 0
    exact = case["clip"] == 0.0
    for step in range(1, STEPS + 1):
        micro = [_grads(case, step, mb, o_scale) for mb in range(case["k"])]
        bad = case["bad"]
        if bad is not None and bad["step"] == step:
            micro[bad["micro"]][bad["rank"]][bad["index"]] = bad["value"]
        if case["k"] > 1:
            res = opt.step_accumulated([[g.to(dev) for g in mb] for mb in micro])
            ores = oracle_mod.zero_step_accum([[_np(g) for g in mb] for mb in micro],
                                              ref["master"], ref["m"], ref["v"], ref["w"], hp,
                                              o_t + 1, o_scale, case["skip"])
        else:
            if graph is not None:
                for b, g in zip(bufs, micro[0]):
                    b.copy_(g)
                graph.replay()
                torch.cuda.synchronize(dev)
                res = opt.last_result()
            else:
                res = opt.step([g.to(dev) for g in micro[0]], api=case["api"])
            ores = oracle_mod.zero_step([_np(g) for g in micro[0]], ref["master"], ref["m"],
                                        ref["v"], ref["w"], hp, o_t + 1, o_scale, case["skip"])
        tag = f"case {case}, step {step}: "
        try:
            compare_result(res, ores)
        except AssertionError as e:
            raise AssertionError(tag + str(e)) from None
        if ores["applied"]:
            o_t += 1
        if case["dynamic"]:
            o_scale, o_good = oracle_mod.loss_scale_update(o_scale, o_good,
                                                           ores["found_nonfinite"], 2, 0.5, 2.0)
        if graph is not None:
            opt.finish_pending()  # the host's t and scale catch up with the device's
        assert opt.t == o_t and opt.scaler.scale == o_scale, tag
        compare_state(state_to_numpy(opt.state()), ref, exact, tag=tag)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_configuration(zero_lib, oracle_mod, seed):
    run_case(draw_case(seed), oracle_mod)


def test_sweep_covers_the_options():
    """The seeds in use reach every option value at least once."""
    cases = [draw_case(s) for s in range(N_CASES)]
    seen = lambda key: {c[key] for c in cases}
    assert seen("dtype") == {"bf16", "fp32"}
    assert {1, 16} <= seen("N") and len(seen("N")) >= 8
    assert seen("k") == {1, 2, 3}
    for key in ("out_of_place", "pingpong", "skip", "dynamic", "device_policy"):
        assert seen(key) == {False, True}, key
    assert seen("staging") == {0, 1} and seen("api") == {"step", "plan"}
    assert {0.0, 0.02, 1.0, 1e6} <= seen("clip")
    assert 0 in seen("bucket") and len(seen("bucket")) > 10
    assert any(c["bad"] is not None and c["skip"] for c in cases)
    assert any(c["bad"] is not None and not c["skip"] for c in cases)
    assert any(c["k"] > 1 and c["staging"] and not c["out_of_place"] for c in cases)
    graphs = [c for c in cases if c["graph"]]
    assert len(graphs) >= 10
    assert {c["out_of_place"] for c in graphs} == {False, True}
    assert {c["staging"] for c in graphs} == {0, 1} and {c["dtype"] for c in graphs} == {"bf16", "fp32"}
    assert any(c["bad"] is not None for c in graphs) and any(c["clip"] > 0 for c in graphs)
    assert sum(c["psi_pad"] > 1 << 22 for c in cases) >= 8
