"""Cases run in a child process against the debug build of the library
(ZERO_GB300_DEBUG=1 loads libzero_gb300_debug.so).  tests/test_gpu_debug_build.py
runs them; this file is not collected by pytest itself.

  parity   a few steps of every kernel form (one-pass register and staged,
           two-pass, accumulation, ping-pong sets, the ZeRO-3 gather) against
           the oracle, bit for bit; the kernels' checks must find nothing.
  sweep    the first 128 configurations of the random parity sweep
           (test_gpu_sweep.py), each against the oracle; the checks must find
           nothing in any of them.
  overrun  with ZERO_DEBUG_TEST_OVERRUN set, the last launch of each pass
           covers groups past the end of the buffers.  Every buffer is
           allocated with a guard region behind it that is larger than the
           overrun, so even an access the checks missed would land in this
           process's own memory; the checks must skip every such access,
           count it, end the step with ZERO_ERR_BOUNDS and leave every guard
           as it was.
"""
from __future__ import annotations

import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
sys.path.insert(0, ROOT)
sys.path.insert(0, HERE)

GUARD = 16384          # elements behind every buffer (the overrun is at most 8192)


def _grads(N, psi, psi_pad, dtype, seed, scale=1024.0):
    g = torch.Generator().manual_seed(seed)
    out = []
    for _ in range(N):
        z = torch.zeros(psi_pad)
        z[:psi] = torch.randn(psi, generator=g) * 1e-3 * scale
        out.append(z.to(torch.bfloat16) if dtype == "bf16" else z)
    return out


def _np(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def parity() -> None:
    import oracle
    from parity_util import compare_result, compare_state, state_to_numpy
    from zero_sharded_mixed_04_gb300 import zero as Z
    from zero_sharded_mixed_04_gb300.optim import ZeroAdam, Zero3Views
    assert Z.DEBUG_BUILD and Z.LIB_PATH.endswith("libzero_gb300_debug.so")
    oracle.build()
    dev = torch.device("cuda:0")
    forms = [dict(), dict(out_of_place=True, skip=True, staging=1),
             dict(out_of_place=True, skip=True, staging=1, policy=True, pingpong=True),
             dict(skip=True), dict(clip=0.5, out_of_place=True, bucket=65_536),
             dict(micro=3, out_of_place=True), dict(micro=2, skip=True)]
    for N, dtype in ((4, "bf16"), (3, "fp32"), (8, "bf16")):
        psi = 200_003
        psi_pad = -(-psi // (N * 128)) * (N * 128)
        for f in forms:
            master = torch.zeros(psi_pad)
            master[:psi] = torch.randn(psi, generator=torch.Generator().manual_seed(N)) * 0.02
            k = f.get("micro", 0)
            opt = ZeroAdam(psi_pad, N, dtype, max_grad_norm=f.get("clip", 0.0),
                           skip_on_overflow=f.get("skip", False), bucket_elems=f.get("bucket", 0),
                           loss_scale=1024.0, out_of_place=f.get("out_of_place", False),
                           device=dev, master=master.to(dev), smem_staging=f.get("staging", 0),
                           micro_batches=k, device_policy=f.get("policy", False),
                           pingpong=f.get("pingpong", False))
            ref = {"master": master.numpy().copy(), "m": np.zeros(psi_pad, np.float32),
                   "v": np.zeros(psi_pad, np.float32), "w": np.zeros(psi_pad, np.uint16)}
            hp = oracle.Hparams(max_grad_norm=f.get("clip", 0.0))
            t = 0
            for step in (1, 2, 3):
                if k:
                    micro = [_grads(N, psi, psi_pad, dtype, 100 * step + mb) for mb in range(k)]
                    if step == 2 and f.get("skip"):
                        micro[1][0][999] = float("inf")
                    res = opt.step_accumulated([[g.to(dev) for g in mb] for mb in micro])
                    ores = oracle.zero_step_accum([[_np(g) for g in mb] for mb in micro],
                                                  ref["master"], ref["m"], ref["v"], ref["w"], hp,
                                                  t + 1, 1024.0, f.get("skip", False))
                else:
                    grads = _grads(N, psi, psi_pad, dtype, step)
                    if step == 2 and f.get("skip"):
                        grads[N - 1][777] = float("inf")
                    res = opt.step([g.to(dev) for g in grads])
                    ores = oracle.zero_step([_np(g) for g in grads], ref["master"], ref["m"],
                                            ref["v"], ref["w"], hp, t + 1, 1024.0,
                                            f.get("skip", False))
                compare_result(res, ores)
                if ores["applied"]:
                    t += 1
                compare_state(state_to_numpy(opt.state()), ref, exact=f.get("clip", 0.0) == 0.0,
                              tag=f"debug build, N={N} {dtype} {f} step {step} ")
        # the ZeRO-3 gather from the last state's shards
        w = opt.state()["w"]
        S = psi_pad // N
        views = Zero3Views([w[r * S:(r + 1) * S] for r in range(N)], S,
                           [(0, 1000), (1000, 77_777), (77_777, psi_pad)], device=dev)
        got = {}
        views.run(lambda i, v: got.__setitem__(i, v.clone()))
        torch.cuda.synchronize()
        full = w.cpu()
        for i, (b, e) in enumerate(views.layers):
            assert torch.equal(got[i].cpu(), full[b:e])
    n = Z.zero_debug_bounds_violations()
    assert n == 0, f"the debug build's checks skipped {n} accesses in correct runs"
    print("debug build parity: ok")


def _guarded(n, dtype, dev, fill):
    """A tensor of n + GUARD elements whose first n are the buffer and whose
    tail is a guard region holding ``fill``."""
    t = torch.empty(n + GUARD, dtype=dtype, device=dev)
    t[n:].fill_(fill)
    return t


def overrun() -> None:
    from zero_sharded_mixed_04_gb300 import zero as Z
    assert Z.DEBUG_BUILD
    overrun_groups = int(os.environ["ZERO_DEBUG_TEST_OVERRUN"])
    assert 0 < overrun_groups * 8 <= GUARD // 2
    dev = torch.device("cuda:0")
    N, psi_pad = 4, 4 * 128 * 300
    cases = [("one pass in place", dict(), False),
             ("one pass out of place", dict(skip_on_overflow=True), True),
             ("staged out of place", dict(skip_on_overflow=True), True),
             ("staged, ping-pong sets", dict(skip_on_overflow=True), True),
             ("two passes (clip)", dict(max_grad_norm=1.0), False),
             ("accumulation", dict(micro_batches=2), True)]
    Z.zero_debug_bounds_violations()   # start from a zero count
    for name, hpkw, out_of_place in cases:
        grads = [_guarded(psi_pad, torch.bfloat16, dev, 3.0) for _ in range(N)]
        for g in grads:
            g[:psi_pad].normal_(0, 1e-3)
        sets = []
        for _ in range(2 if out_of_place else 1):
            sets.append({"master": _guarded(psi_pad, torch.float32, dev, 7.0),
                         "m": _guarded(psi_pad, torch.float32, dev, 7.0),
                         "v": _guarded(psi_pad, torch.float32, dev, 7.0),
                         "w": _guarded(psi_pad, torch.int16, dev, 77)})
            for k in ("master", "m", "v"):
                sets[-1][k][:psi_pad].zero_()
            sets[-1]["w"][:psi_pad].zero_()
        hp = Z.make_hparams(**hpkw)
        src, dst = sets[0], sets[-1]
        ws_bytes = Z.zero_workspace_bytes(psi_pad, hp, not out_of_place)
        ws = torch.zeros(ws_bytes + 4 * GUARD, dtype=torch.uint8, device=dev)
        ws[ws_bytes:].fill_(99)
        before = {id(t): t.clone() for s in sets for t in s.values()}
        before.update({id(g): g.clone() for g in grads})
        res = torch.zeros(4, dtype=torch.int32, pin_memory=True)
        word = torch.zeros(1, dtype=torch.int32, pin_memory=True)
        plan = Z.zero_plan()
        view = lambda t: t[:psi_pad]
        rc = Z.zero_plan_init(plan, [view(g) for g in grads], Z.ZERO_GRAD_BF16,
                              *[view(src[k]) for k in ("master", "m", "v", "w")],
                              *[view(dst[k]) for k in ("master", "m", "v", "w")],
                              psi_pad, N, hp, 1.0, ws, ws_bytes)
        assert rc == Z.ZERO_OK, (name, rc)
        if "staged" in name:
            plan.smem_staging = Z.ZERO_STAGING_TMA
        if "ping-pong" in name:
            assert Z.zero_plan_set_pingpong(plan, word) == Z.ZERO_OK
        assert Z.zero_plan_begin(plan, None) == Z.ZERO_OK
        for _ in range(max(1, hp.micro_batches)):
            assert Z.zero_plan_bucket(plan, 0, psi_pad, None, None) == Z.ZERO_OK
        assert Z.zero_plan_end(plan, res, None) == Z.ZERO_OK
        torch.cuda.synchronize()
        status = int(res[0])
        n = Z.zero_debug_bounds_violations()
        assert status == Z.ZERO_ERR_BOUNDS, (name, status)
        assert n > 0, (name, n)
        for s in sets:
            for k, t in s.items():
                assert torch.equal(t[psi_pad:], before[id(t)][psi_pad:]), (name, k, "guard written")
        for g in grads:
            assert torch.equal(g, before[id(g)]), (name, "gradients written")
        assert torch.equal(ws[ws_bytes:], torch.full_like(ws[ws_bytes:], 99)), (name, "workspace guard")
        if "ping-pong" in name:
            assert int(word[0]) == 0, "a step that hit the checks must not change the current set"
        elif out_of_place:
            # a step that hit the checks is not applied: dst holds src again
            for k in ("master", "m", "v", "w"):
                assert torch.equal(view(dst[k]), view(src[k])), (name, k)
    # the ZeRO-3 gather: the last segment is made longer than the range
    shard = 4096
    shards = [_guarded(shard, torch.int16, dev, 5) for _ in range(N)]
    for r, x in enumerate(shards):
        x[:shard] = r + 1
    view = _guarded(3 * shard, torch.int16, dev, 55)
    assert Z.zero3_gather([x[:shard] for x in shards], N, shard, 0, 3 * shard,
                          view[:3 * shard]) == Z.ZERO_OK
    torch.cuda.synchronize()
    assert Z.zero_debug_bounds_violations() > 0
    assert torch.equal(view[3 * shard:], torch.full_like(view[3 * shard:], 55)), "view guard"
    print("debug build overrun: ok")


def sweep() -> None:
    import oracle
    from test_gpu_sweep import draw_case, run_case
    from zero_sharded_mixed_04_gb300 import zero as Z
    assert Z.DEBUG_BUILD and Z.LIB_PATH.endswith("libzero_gb300_debug.so")
    oracle.build()
    for seed in range(128):
        run_case(draw_case(seed), oracle)
    n = Z.zero_debug_bounds_violations()
    assert n == 0, f"the debug build's checks skipped {n} accesses in the sweep"
    print("debug build sweep: ok")


if __name__ == "__main__":
    {"parity": parity, "overrun": overrun, "sweep": sweep}[sys.argv[1]]()
