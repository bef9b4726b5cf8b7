"""GPU parity: the CUDA path through the C ABI against the oracle, on the same
seeded inputs, element by element, over several steps.

Sizes span several sweeps of the persistent grid plus ragged tails.  The
matrix covers:
  - N = 1..8 and a large N;
  - BF16 and FP32 gradients;
  - in place and out of place;
  - the one-pass and two-pass forms, and buckets;
  - weight decay, clipping, skip on overflow and the dynamic loss scale;
  - non-finite gradients and the degenerate sizes (empty vector, one
    parameter).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from parity_util import compare_result, compare_state, state_to_numpy

pytestmark = pytest.mark.gpu


def _oracle_state(master_np):
    n = master_np.size
    return {"master": master_np.copy(), "m": np.zeros(n, np.float32), "v": np.zeros(n, np.float32),
            "w": np.zeros(n, np.uint16)}


def _make_grads(N, psi, psi_pad, dtype, sigma, seed, gen_device="cpu"):
    g = torch.Generator(device=gen_device)
    g.manual_seed(seed)
    out = []
    for _ in range(N):
        z = torch.zeros(psi_pad, dtype=torch.float32)
        z[:psi] = torch.randn(psi, generator=g) * sigma
        out.append(z.to(torch.bfloat16) if dtype == "bf16" else z)
    return out


def _np(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def run_parity(zero_lib, oracle_mod, *, N, psi, dtype="bf16", steps=3, lr=1e-3, wd=0.0,
               clip=0.0, skip=False, out_of_place=False, bucket=0, loss_scale=1.0,
               dynamic=False, growth_interval=2000, sigma=1e-3, bad_step=0, bad_value=np.inf,
               seed=1234, api="step", per_bucket_events=False, host_accum=False, staging=0,
               device_policy=False, pingpong=False):
    from zero_sharded_mixed_04_gb300.optim import ZeroAdam
    dev = torch.device("cuda:0")
    unit = N * 128
    psi_pad = -(-psi // unit) * unit
    gm = torch.Generator()
    gm.manual_seed(seed)
    master = torch.zeros(psi_pad, dtype=torch.float32)
    master[:psi] = torch.randn(psi, generator=gm) * 0.02
    opt = ZeroAdam(psi_pad, N, dtype, lr=lr, weight_decay=wd, max_grad_norm=clip,
                   skip_on_overflow=skip, bucket_elems=bucket, loss_scale=loss_scale,
                   dynamic_loss_scale=dynamic, growth_interval=growth_interval,
                   out_of_place=out_of_place, device=dev, master=master.to(dev),
                   host_grad_accum=host_accum, smem_staging=staging, device_policy=device_policy,
                   pingpong=pingpong)
    ref = _oracle_state(master.numpy())
    hp = oracle_mod.Hparams(lr=lr, weight_decay=wd, max_grad_norm=clip)
    o_t, o_scale, o_good = 0, loss_scale, 0
    exact = clip == 0.0
    for step in range(1, steps + 1):
        grads = _make_grads(N, psi, psi_pad, dtype, sigma * o_scale, seed + step)
        if step == bad_step and psi > 0:
            grads[N - 1][min(psi - 1, 12345)] = float(bad_value)
        ev = None
        if per_bucket_events:
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in opt.bucket_bounds()]
        res = opt.step([g.to(dev) for g in grads], api=api, bucket_events=ev)
        ores = oracle_mod.zero_step([_np(g) for g in grads], ref["master"], ref["m"], ref["v"],
                                    ref["w"], hp, o_t + 1, o_scale, skip)
        compare_result(res, ores)
        if ores["applied"]:
            o_t += 1
        if dynamic:
            o_scale, o_good = oracle_mod.loss_scale_update(o_scale, o_good,
                                                           ores["found_nonfinite"],
                                                           growth_interval, 0.5, 2.0)
        assert opt.t == o_t and opt.scaler.scale == o_scale
        compare_state(state_to_numpy(opt.state()), ref, exact, tag=f"step {step} ")
    return opt, ref


PSI_MULTI_SWEEP = 3_000_017   # several sweeps of the persistent grid, ragged tail
PSI_SMALL = 200_003


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_one_pass_in_place(zero_lib, oracle_mod, N, dtype):
    psi = PSI_MULTI_SWEEP if N in (4, 8) else PSI_SMALL
    run_parity(zero_lib, oracle_mod, N=N, psi=psi, dtype=dtype)


@pytest.mark.parametrize("N,dtype", [(4, "bf16"), (3, "fp32"), (8, "bf16")])
def test_adamw_weight_decay(zero_lib, oracle_mod, N, dtype):
    run_parity(zero_lib, oracle_mod, N=N, psi=PSI_SMALL, dtype=dtype, wd=0.1, steps=4)


@pytest.mark.parametrize("out_of_place", [False, True])
@pytest.mark.parametrize("N,dtype", [(4, "bf16"), (8, "bf16"), (4, "fp32"), (5, "bf16")])
def test_skip_on_overflow(zero_lib, oracle_mod, N, dtype, out_of_place):
    """Step 2 gets one +inf; with the skip on it must leave the state
    bit-unchanged and the next steps continue from there."""
    run_parity(zero_lib, oracle_mod, N=N, psi=PSI_MULTI_SWEEP if N == 8 else PSI_SMALL,
               dtype=dtype, steps=4, skip=True, out_of_place=out_of_place, bad_step=2,
               loss_scale=1024.0, dynamic=True)


@pytest.mark.parametrize("bad", [np.inf, -np.inf, np.nan])
@pytest.mark.parametrize("out_of_place", [False, True])
def test_nonfinite_values(zero_lib, oracle_mod, bad, out_of_place):
    run_parity(zero_lib, oracle_mod, N=4, psi=PSI_SMALL, steps=3, skip=True,
               out_of_place=out_of_place, bad_step=1, bad_value=bad)


def test_nonfinite_without_skip_propagates(zero_lib, oracle_mod):
    run_parity(zero_lib, oracle_mod, N=4, psi=PSI_SMALL, steps=2, skip=False, bad_step=1)


@pytest.mark.parametrize("out_of_place", [False, True])
@pytest.mark.parametrize("N,dtype,clip", [(4, "fp32", 1.0), (4, "bf16", 0.01), (8, "bf16", 1e-4),
                                          (3, "fp32", 1e9)])
def test_global_norm_clip(zero_lib, oracle_mod, N, dtype, clip, out_of_place):
    run_parity(zero_lib, oracle_mod, N=N, psi=PSI_MULTI_SWEEP if N == 8 else PSI_SMALL,
               dtype=dtype, clip=clip, out_of_place=out_of_place, steps=3)


@pytest.mark.parametrize("out_of_place", [False, True])
def test_clip_with_skip(zero_lib, oracle_mod, out_of_place):
    run_parity(zero_lib, oracle_mod, N=4, psi=PSI_SMALL, clip=0.5, skip=True,
               out_of_place=out_of_place, bad_step=2, steps=3)


@pytest.mark.parametrize("bucket", [8, 262_248, 1_000_000])
@pytest.mark.parametrize("out_of_place,skip", [(False, False), (False, True), (True, True)])
def test_buckets(zero_lib, oracle_mod, bucket, out_of_place, skip):
    psi = PSI_SMALL if bucket == 8 else PSI_MULTI_SWEEP
    run_parity(zero_lib, oracle_mod, N=8, psi=psi if bucket != 8 else 20_000, bucket=bucket,
               out_of_place=out_of_place, skip=skip, steps=2, loss_scale=65536.0,
               dynamic=True, bad_step=2 if skip else 0)


def test_dynamic_loss_scale_growth(zero_lib, oracle_mod):
    run_parity(zero_lib, oracle_mod, N=2, psi=20_000, steps=7, skip=True, out_of_place=True,
               loss_scale=256.0, dynamic=True, growth_interval=2, bad_step=4)


@pytest.mark.parametrize("psi", [1, 127, 128, 129, 1023])
def test_tiny_and_ragged(zero_lib, oracle_mod, psi):
    run_parity(zero_lib, oracle_mod, N=4, psi=psi, steps=2)
    run_parity(zero_lib, oracle_mod, N=3, psi=psi, steps=2, dtype="fp32", clip=1e-3)


def test_many_ranks(zero_lib, oracle_mod):
    run_parity(zero_lib, oracle_mod, N=64, psi=100_000, steps=2)
    run_parity(zero_lib, oracle_mod, N=13, psi=100_000, steps=2, dtype="fp32", skip=True,
               bad_step=2)


def test_empty_vector(zero_lib):
    Z = zero_lib
    hp = Z.make_hparams(skip_on_overflow=True)
    ws = torch.empty(Z.zero_workspace_bytes(0, hp, True), dtype=torch.uint8, device="cuda")
    rc = Z.zero_step([None, None], Z.ZERO_GRAD_BF16, None, None, None, None, 0, 2, hp, 1.0, ws,
                     ws.numel(), None, None)
    assert rc == Z.ZERO_OK


def test_blocking_call_returns_status(zero_lib):
    """With no result pointer the call waits and returns the step status."""
    Z = zero_lib
    dev = torch.device("cuda:0")
    N, n = 2, 2 * 128 * 4
    grads = [torch.zeros(n, dtype=torch.bfloat16, device=dev) for _ in range(N)]
    grads[1][5] = float("nan")
    st = [torch.zeros(n, dtype=torch.float32, device=dev) for _ in range(3)]
    w = torch.zeros(n, dtype=torch.int16, device=dev)
    hp = Z.make_hparams(skip_on_overflow=True)
    ws = torch.empty(Z.zero_workspace_bytes(n, hp, True), dtype=torch.uint8, device=dev)
    rc = Z.zero_step(grads, Z.ZERO_GRAD_BF16, *st, w, n, N, hp, 1.0, ws, ws.numel(), None, None)
    assert rc == Z.ZERO_STEP_SKIPPED
    grads[1][5] = 0.0
    rc = Z.zero_step(grads, Z.ZERO_GRAD_BF16, *st, w, n, N, hp, 1.0, ws, ws.numel(), None, None)
    assert rc == Z.ZERO_OK


def test_launch_count_grows(zero_lib):
    Z = zero_lib
    before = Z.zero_launch_count()
    test_blocking_call_returns_status(zero_lib)
    assert Z.zero_launch_count() >= before + 4


@pytest.mark.parametrize("out_of_place,skip,clip", [(False, False, 0.0), (True, True, 0.0),
                                                   (False, True, 0.0), (True, False, 0.3)])
@pytest.mark.parametrize("per_bucket_events", [False, True])
def test_plan_api(zero_lib, oracle_mod, out_of_place, skip, clip, per_bucket_events):
    """The bucketed entry points give the same result as zero_step, with
    consecutive bucket launches overlapping (nothing enqueued between them)
    and without (events recorded between them)."""
    run_parity(zero_lib, oracle_mod, N=8, psi=PSI_MULTI_SWEEP, bucket=400_000,
               out_of_place=out_of_place, skip=skip, clip=clip, steps=3, api="plan",
               bad_step=2 if skip else 0, loss_scale=4096.0, dynamic=skip,
               per_bucket_events=per_bucket_events)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_plan_two_staging_slots(zero_lib, oracle_mod, dtype):
    """Gradients streamed bucket by bucket through two device slots (one in
    use while the other loads) give the state the whole-vector step gives."""
    Z = zero_lib
    dev = torch.device("cuda:0")
    N, psi, bucket = 4, 1_000_003, 131_072
    psi_pad = -(-psi // (N * 128)) * (N * 128)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    grads = _make_grads(N, psi, psi_pad, dtype, 1e-3, 99)
    host = [g.pin_memory() for g in grads]
    master = torch.randn(psi_pad, generator=torch.Generator().manual_seed(5)) * 0.02
    master[psi:] = 0
    st = {k: torch.zeros(psi_pad, dtype=torch.float32, device=dev) for k in ("m", "v")}
    st["master"] = master.to(dev)
    w = torch.zeros(psi_pad, dtype=torch.int16, device=dev)
    hp = Z.make_hparams(skip_on_overflow=False)
    ws = torch.empty(Z.zero_workspace_bytes(psi_pad, hp, True), dtype=torch.uint8, device=dev)
    slots = [[torch.empty(bucket, dtype=tdt, device=dev) for _ in range(N)] for _ in range(2)]
    compute = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    freed = [torch.cuda.Event(), torch.cuda.Event()]
    loaded = [torch.cuda.Event(), torch.cuda.Event()]
    plan = Z.zero_plan()
    assert Z.zero_plan_init(plan, [None] * N, Z.ZERO_GRAD_BF16 if dtype == "bf16" else
                            Z.ZERO_GRAD_FP32, st["master"], st["m"], st["v"], w, st["master"],
                            st["m"], st["v"], w, psi_pad, N, hp, 1.0, ws, ws.numel()) == 0
    assert Z.zero_plan_begin(plan, compute) == 0
    for k, b0 in enumerate(range(0, psi_pad, bucket)):
        b1 = min(psi_pad, b0 + bucket)
        slot = k % 2
        with torch.cuda.stream(copy):
            copy.wait_event(freed[slot])
            for i in range(N):
                slots[slot][i][:b1 - b0].copy_(host[i][b0:b1], non_blocking=True)
            loaded[slot].record(copy)
        compute.wait_event(loaded[slot])
        assert Z.zero_plan_bucket(plan, b0, b1, [t for t in slots[slot]], compute) == 0
        freed[slot].record(compute)
    res = Z.zero_step_result()
    res_t = torch.zeros(4, dtype=torch.int32, pin_memory=True)
    assert Z.zero_plan_end(plan, res_t, compute) == 0
    torch.cuda.synchronize()
    ref = _oracle_state(master.numpy())
    ores = oracle_mod.zero_step([_np(g) for g in grads], ref["master"], ref["m"], ref["v"],
                                ref["w"], oracle_mod.Hparams(), 1, 1.0, False)
    assert int(res_t[0]) == 0 and ores["applied"]
    got = {"master": st["master"].cpu().numpy(), "m": st["m"].cpu().numpy(),
           "v": st["v"].cpu().numpy(), "w": w.cpu().numpy().view(np.uint16)}
    compare_state(got, ref, exact=True)


def test_async_steps_without_host_reads(zero_lib, oracle_mod):
    """With no skip and a static loss scale, steps are enqueued back to back
    without reading their outcome; the state after them matches the oracle."""
    from zero_sharded_mixed_04_gb300.optim import ZeroAdam
    dev = torch.device("cuda:0")
    N, psi = 4, PSI_MULTI_SWEEP
    psi_pad = -(-psi // (N * 128)) * (N * 128)
    master = torch.zeros(psi_pad)
    master[:psi] = torch.randn(psi, generator=torch.Generator().manual_seed(3)) * 0.02
    opt = ZeroAdam(psi_pad, N, "bf16", weight_decay=0.1, bucket_elems=1_000_000, device=dev,
                   master=master.to(dev))
    assert not opt.needs_result
    ref = _oracle_state(master.numpy())
    hp = oracle_mod.Hparams(weight_decay=0.1)
    all_grads = [_make_grads(N, psi, psi_pad, "bf16", 1e-3, 500 + s) for s in range(4)]
    dev_grads = [[g.to(dev) for g in gs] for gs in all_grads]
    for s, gs in enumerate(dev_grads):
        assert opt.step_async(gs, api="plan" if s % 2 else "step") is None
    assert opt.t == 4
    for s, gs in enumerate(all_grads):
        ores = oracle_mod.zero_step([_np(g) for g in gs], ref["master"], ref["m"], ref["v"],
                                    ref["w"], hp, s + 1, 1.0, False)
    compare_result(opt.last_result(), ores)
    compare_state(state_to_numpy(opt.state()), ref, exact=True)


ACCUMULATION_CASES = [
    (4, 2, "bf16", 0.0, False, False, 0, 0.0),
    (8, 3, "bf16", 0.0, True, True, 400_000, 0.0),
    (3, 4, "fp32", 0.05, False, False, 262_144, 0.1),
    (2, 2, "fp32", 0.0, True, False, 0, 0.1),
    (4, 5, "bf16", 1.0, True, True, 1_000_000, 0.0),
    (2, 3, "fp32", 0.0, False, True, 0, 0.1),
    (5, 2, "fp32", 0.0, True, True, 262_144, 0.0),
]


def run_accumulation(zero_lib, oracle_mod, N, k, dtype, clip, skip, out_of_place, bucket, wd,
                     staging=0):
    """k micro-batches reduce-scattered bucket by bucket into the owner's FP32
    accumulator, then one update; against the oracle's accumulation.  With
    the skip on, micro-batch 1 of step 2 carries a +inf."""
    from zero_sharded_mixed_04_gb300.optim import ZeroAdam
    dev = torch.device("cuda:0")
    psi = PSI_MULTI_SWEEP if N >= 4 else PSI_SMALL
    psi_pad = -(-psi // (N * 128)) * (N * 128)
    master = torch.zeros(psi_pad)
    master[:psi] = torch.randn(psi, generator=torch.Generator().manual_seed(11)) * 0.02
    opt = ZeroAdam(psi_pad, N, dtype, weight_decay=wd, max_grad_norm=clip, skip_on_overflow=skip,
                   bucket_elems=bucket, loss_scale=256.0, out_of_place=out_of_place, device=dev,
                   master=master.to(dev), micro_batches=k, smem_staging=staging)
    ref = _oracle_state(master.numpy())
    hp = oracle_mod.Hparams(weight_decay=wd, max_grad_norm=clip)
    o_t = 0
    for step in range(1, 4):
        micro = [_make_grads(N, psi, psi_pad, dtype, 1e-3 * 256.0, 1000 * step + mb)
                 for mb in range(k)]
        if skip and step == 2:
            micro[1][N - 1][777] = float("inf")
        res = opt.step_accumulated([[g.to(dev) for g in mb] for mb in micro])
        ores = oracle_mod.zero_step_accum([[_np(g) for g in mb] for mb in micro], ref["master"],
                                          ref["m"], ref["v"], ref["w"], hp, o_t + 1, 256.0, skip)
        compare_result(res, ores)
        if ores["applied"]:
            o_t += 1
        assert opt.t == o_t
        compare_state(state_to_numpy(opt.state()), ref, exact=clip == 0.0, tag=f"step {step} ")
    if skip:
        assert o_t == 2


@pytest.mark.parametrize("N,k,dtype,clip,skip,out_of_place,bucket,wd", ACCUMULATION_CASES)
def test_gradient_accumulation(zero_lib, oracle_mod, N, k, dtype, clip, skip, out_of_place,
                               bucket, wd):
    """Without clip, and unless an in-place step may be skipped, the last
    micro-batch is added and applied in one pass (the first, second, sixth and
    seventh cases; in the seventh the +inf arrives in that last micro-batch)."""
    run_accumulation(zero_lib, oracle_mod, N, k, dtype, clip, skip, out_of_place, bucket, wd)



@pytest.mark.parametrize("N,dtype,skip,clip,out_of_place,bucket", [
    (4, "bf16", True, 0.0, False, 0),          # two passes because of the in-place skip
    (8, "bf16", False, 0.0, True, 400_000),     # forced to two passes by the host shard
    (4, "fp32", False, 0.5, True, 0),           # clip
])
def test_gradient_shard_in_host_memory(zero_lib, oracle_mod, N, dtype, skip, clip, out_of_place,
                                       bucket):
    """The owner's FP32 combined gradient kept in pinned host memory and reached
    over the host link: the same step, bit for bit (within the clip tolerance)."""
    run_parity(zero_lib, oracle_mod, N=N, psi=PSI_MULTI_SWEEP if N == 8 else PSI_SMALL,
               dtype=dtype, skip=skip, clip=clip, out_of_place=out_of_place, bucket=bucket,
               steps=3, bad_step=2 if skip else 0, loss_scale=512.0, dynamic=skip,
               host_accum=True)


def test_host_shard_accumulation_through_two_slots(zero_lib, oracle_mod):
    """Gradients in pinned host memory stream through two device slots; each
    reduced bucket is added to the owner's FP32 shard in host memory; the GPU
    keeps no gradient shard (the offloaded-shard pattern with two buffers)."""
    from zero_sharded_mixed_04_gb300.optim import ZeroAdam
    dev = torch.device("cuda:0")
    N, psi, bucket = 8, PSI_MULTI_SWEEP, 400_000
    psi_pad = -(-psi // (N * 128)) * (N * 128)
    master = torch.zeros(psi_pad)
    master[:psi] = torch.randn(psi, generator=torch.Generator().manual_seed(21)) * 0.02
    opt = ZeroAdam(psi_pad, N, "bf16", bucket_elems=bucket, skip_on_overflow=True,
                   out_of_place=True, loss_scale=1024.0, device=dev, master=master.to(dev),
                   host_grad_accum=True)
    assert opt.ws_bytes == zero_lib.ZERO_WORKSPACE_CONTROL_BYTES
    slots = opt.make_slots()
    copy_stream = torch.cuda.Stream(dev)
    ref = _oracle_state(master.numpy())
    hp = oracle_mod.Hparams()
    for step in (1, 2):
        grads = _make_grads(N, psi, psi_pad, "bf16", 1e-3 * 1024.0, 77 + step)
        host = [g.pin_memory() for g in grads]
        opt.enqueue_from_host(host, slots, copy_stream)
        res = opt.finish()
        ores = oracle_mod.zero_step([_np(g) for g in grads], ref["master"], ref["m"], ref["v"],
                                    ref["w"], hp, step, 1024.0, True)
        compare_result(res, ores)
        compare_state(state_to_numpy(opt.state()), ref, exact=True, tag=f"step {step} ")
        # the host shard holds this step's combined gradient
        g_host = opt.grad_accum.numpy()
        g_ref = oracle_mod.all_reduce([_np(g) for g in grads], psi_pad, np.float32(1 / (8 * 1024.0)))
        assert np.array_equal(g_host.view(np.uint32), g_ref.view(np.uint32))


def test_host_shard_gradient_accumulation(zero_lib, oracle_mod):
    from zero_sharded_mixed_04_gb300.optim import ZeroAdam
    dev = torch.device("cuda:0")
    N, k, psi = 4, 3, PSI_SMALL
    psi_pad = -(-psi // (N * 128)) * (N * 128)
    master = torch.zeros(psi_pad)
    master[:psi] = torch.randn(psi, generator=torch.Generator().manual_seed(5)) * 0.02
    opt = ZeroAdam(psi_pad, N, "bf16", bucket_elems=65_536, device=dev, master=master.to(dev),
                   micro_batches=k, host_grad_accum=True)
    ref = _oracle_state(master.numpy())
    for step in (1, 2):
        micro = [_make_grads(N, psi, psi_pad, "bf16", 1e-3, 300 * step + mb) for mb in range(k)]
        res = opt.step_accumulated([[g.to(dev) for g in mb] for mb in micro])
        ores = oracle_mod.zero_step_accum([[_np(g) for g in mb] for mb in micro], ref["master"],
                                          ref["m"], ref["v"], ref["w"], oracle_mod.Hparams(),
                                          step, 1.0, False)
        compare_result(res, ores)
        compare_state(state_to_numpy(opt.state()), ref, exact=True, tag=f"step {step} ")


def _policy_run(zero_lib, oracle_mod, *, out_of_place, skip, bad_steps, steps, async_steps,
                N=4, psi=PSI_SMALL, clip=0.0, pingpong=False, staging=0):
    from zero_sharded_mixed_04_gb300.optim import ZeroAdam
    dev = torch.device("cuda:0")
    psi_pad = -(-psi // (N * 128)) * (N * 128)
    master = torch.zeros(psi_pad)
    master[:psi] = torch.randn(psi, generator=torch.Generator().manual_seed(8)) * 0.02
    opt = ZeroAdam(psi_pad, N, "bf16", skip_on_overflow=skip, max_grad_norm=clip,
                   loss_scale=4096.0, dynamic_loss_scale=True, growth_interval=2,
                   out_of_place=out_of_place, device=dev, master=master.to(dev),
                   device_policy=True, pingpong=pingpong, smem_staging=staging)
    assert not opt.needs_result
    ref = _oracle_state(master.numpy())
    hp = oracle_mod.Hparams(max_grad_norm=clip)
    o_t, o_scale, o_good = 0, 4096.0, 0
    all_grads = []
    for step in range(1, steps + 1):
        # every step's gradients are drawn at the oracle's running scale, which
        # the device policy must track too
        grads = _make_grads(N, psi, psi_pad, "bf16", 1e-3 * o_scale, 900 + step)
        if step in bad_steps:
            grads[1][4321] = float("inf")
        all_grads.append(grads)
        ores = oracle_mod.zero_step([_np(g) for g in grads], ref["master"], ref["m"], ref["v"],
                                    ref["w"], hp, o_t + 1, o_scale, skip)
        if ores["applied"]:
            o_t += 1
        o_scale, o_good = oracle_mod.loss_scale_update(o_scale, o_good, ores["found_nonfinite"],
                                                       2, 0.5, 2.0)
    dev_grads = [[g.to(dev) for g in gs] for gs in all_grads]
    torch.cuda.synchronize()
    for step, gs in enumerate(dev_grads, start=1):
        if async_steps:
            assert opt.step_async(gs) is None
        else:
            opt.step(gs)
    res = opt.finish()
    assert res["status"] in (zero_lib.ZERO_OK, zero_lib.ZERO_STEP_SKIPPED)
    assert opt.t == o_t and opt.scaler.scale == o_scale
    compare_state(state_to_numpy(opt.state()), ref, exact=clip == 0.0)


@pytest.mark.parametrize("out_of_place", [False, True])
def test_accumulation_with_device_policy(zero_lib, oracle_mod, out_of_place):
    """Micro-batch accumulation with t and the dynamic loss scale kept on the
    device, steps enqueued back to back: step 3 overflows in its last
    micro-batch and step 4 in its first, and both are skipped.  Out of place
    the last micro-batch is added and applied in one pass; in place it takes
    the second pass."""
    from zero_sharded_mixed_04_gb300.optim import ZeroAdam
    dev = torch.device("cuda:0")
    N, k, psi, steps = 4, 3, PSI_SMALL, 6
    psi_pad = -(-psi // (N * 128)) * (N * 128)
    master = torch.zeros(psi_pad)
    master[:psi] = torch.randn(psi, generator=torch.Generator().manual_seed(13)) * 0.02
    opt = ZeroAdam(psi_pad, N, "bf16", skip_on_overflow=True, bucket_elems=131_072,
                   loss_scale=4096.0, dynamic_loss_scale=True, growth_interval=2,
                   out_of_place=out_of_place, device=dev, master=master.to(dev),
                   micro_batches=k, device_policy=True)
    assert not opt.needs_result
    ref = _oracle_state(master.numpy())
    hp = oracle_mod.Hparams()
    o_t, o_scale, o_good = 0, 4096.0, 0
    all_micro = []
    for step in range(1, steps + 1):
        micro = [_make_grads(N, psi, psi_pad, "bf16", 1e-3 * o_scale, 700 * step + mb)
                 for mb in range(k)]
        if step == 3:
            micro[k - 1][2][999] = float("inf")
        if step == 4:
            micro[0][0][5] = float("-inf")
        all_micro.append(micro)
        ores = oracle_mod.zero_step_accum([[_np(g) for g in mb] for mb in micro], ref["master"],
                                          ref["m"], ref["v"], ref["w"], hp, o_t + 1, o_scale,
                                          True)
        if ores["applied"]:
            o_t += 1
        o_scale, o_good = oracle_mod.loss_scale_update(o_scale, o_good, ores["found_nonfinite"],
                                                       2, 0.5, 2.0)
    dev_micro = [[[g.to(dev) for g in mb] for mb in micro] for micro in all_micro]
    torch.cuda.synchronize()
    for micro in dev_micro:
        opt.enqueue_accumulated(micro)
    res = opt.finish()
    assert res["status"] == zero_lib.ZERO_OK
    assert o_t == steps - 2
    assert opt.t == o_t and opt.scaler.scale == o_scale
    compare_state(state_to_numpy(opt.state()), ref, exact=True)


@pytest.mark.parametrize("out_of_place", [False, True])
@pytest.mark.parametrize("async_steps", [False, True])
def test_device_policy_tracks_the_host_rule(zero_lib, oracle_mod, out_of_place, async_steps):
    """t and the dynamic loss scale kept on the device: steps issued with
    (step by step) or without (back to back) host reads give the oracle's
    state, t and scale; steps 3 and 4 overflow and are skipped."""
    _policy_run(zero_lib, oracle_mod, out_of_place=out_of_place, skip=True, bad_steps={3, 4},
                steps=7, async_steps=async_steps)


def test_device_policy_with_clip(zero_lib, oracle_mod):
    _policy_run(zero_lib, oracle_mod, out_of_place=True, skip=True, bad_steps={2}, steps=4,
                async_steps=True, clip=0.05)


@pytest.mark.parametrize("out_of_place", [False, True])
def test_device_policy_window_miss_changes_nothing(zero_lib, out_of_place):
    """A step whose device t falls outside the window it was given leaves the
    state untouched (a copy of it, out of place) and reports the miss."""
    import ctypes
    Z = zero_lib
    dev = torch.device("cuda:0")
    N, n = 4, 4 * 128 * 64
    grads = [(torch.randn(n, generator=torch.Generator().manual_seed(i)) * 1e-3).to(
        torch.bfloat16).to(dev) for i in range(N)]
    src = [torch.randn(n, device=dev) * 0.02, torch.rand(n, device=dev) * 1e-4,
           torch.rand(n, device=dev) * 1e-6, torch.zeros(n, dtype=torch.int16, device=dev)]
    before = [t.clone() for t in src]
    dst = [torch.full_like(t, 7) for t in src] if out_of_place else src
    hp = Z.make_hparams(skip_on_overflow=False)
    ws = torch.empty(Z.zero_workspace_bytes(n, hp, not out_of_place), dtype=torch.uint8,
                     device=dev)
    pol_mem = torch.zeros(ctypes.sizeof(Z.zero_device_policy), dtype=torch.uint8, pin_memory=True)
    pol = Z.zero_device_policy.from_address(pol_mem.data_ptr())
    pol.t, pol.loss_scale = 5, 1.0
    res = torch.zeros(4, dtype=torch.int32, pin_memory=True)
    plan = Z.zero_plan()
    assert Z.zero_plan_init(plan, grads, Z.ZERO_GRAD_BF16, *src, *dst, n, N, hp, 1.0, ws,
                            ws.numel()) == Z.ZERO_OK
    assert Z.zero_plan_set_device_policy(plan, pol_mem, 1, 3) == Z.ZERO_OK   # t' = 6 is outside
    assert Z.zero_plan_begin(plan, None) == Z.ZERO_OK
    assert Z.zero_plan_bucket(plan, 0, n, None, None) == Z.ZERO_OK
    assert Z.zero_plan_end(plan, res, None) == Z.ZERO_OK
    torch.cuda.synchronize()
    assert int(res[0]) == Z.ZERO_ERR_POLICY_WINDOW
    assert pol.t == 5 and pol.last_status == Z.ZERO_ERR_POLICY_WINDOW
    for a, b in zip(dst, before):
        assert torch.equal(a, b)
    for a, b in zip(src, before):
        assert torch.equal(a, b)


def test_host_buffer_is_page_locked_and_huge_page_backed():
    """hostmem.HostBuffer: registered with the driver (torch sees it as pinned),
    asynchronous copies both ways keep the bits, and closing unregisters it."""
    from zero_sharded_mixed_04_gb300.hostmem import HostBuffer
    n = 3 * (1 << 20) + 5
    buf = HostBuffer(n, torch.bfloat16)
    assert buf.kind == "huge-page mapping, cudaHostRegister"
    assert buf.tensor.is_pinned() and buf.tensor.numel() == n
    src = torch.randint(-32768, 32767, (n,), dtype=torch.int16,
                        generator=torch.Generator().manual_seed(4)).view(torch.bfloat16)
    buf.tensor.copy_(src)
    dev = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    dev.copy_(buf.tensor, non_blocking=True)
    back = HostBuffer(n, torch.bfloat16)
    back.tensor.copy_(dev, non_blocking=True)
    torch.cuda.synchronize()
    assert torch.equal(back.tensor.view(torch.int16), src.view(torch.int16))
    buf.close()
    back.close()
    assert buf.tensor is None


# ---------------------------------------------------------------------------
# Ping-pong state sets: the device keeps which of the two out-of-place sets
# is current, so a skipped step copies nothing.

@pytest.mark.parametrize("staging", [0, 1])
@pytest.mark.parametrize("N,dtype", [(4, "bf16"), (8, "bf16"), (3, "fp32")])
def test_pingpong_skip(zero_lib, oracle_mod, N, dtype, staging):
    """Step 2 overflows and is skipped; the current set must stay current and
    the later steps continue from it (host-side bookkeeping)."""
    opt, _ = run_parity(zero_lib, oracle_mod, N=N, psi=PSI_MULTI_SWEEP if N == 8 else PSI_SMALL,
                        dtype=dtype, steps=4, skip=True, out_of_place=True, bad_step=2,
                        loss_scale=1024.0, dynamic=True, staging=staging, pingpong=True)
    # three applied steps flip the set three times
    assert int(opt.set_mem[0]) == 1 and opt.cur == 1


@pytest.mark.parametrize("clip,bucket", [(0.05, 0), (1.0, 400_000)])
def test_pingpong_two_pass(zero_lib, oracle_mod, clip, bucket):
    """With clipping the update runs as a second pass after the step-wide
    decision: it reads the snapshot of the current set, not the flipped word."""
    run_parity(zero_lib, oracle_mod, N=8, psi=PSI_MULTI_SWEEP, dtype="bf16", steps=4, skip=True,
               clip=clip, out_of_place=True, bad_step=3, bucket=bucket, loss_scale=4096.0,
               dynamic=True, pingpong=True)


@pytest.mark.parametrize("staging", [0, 1])
@pytest.mark.parametrize("async_steps", [False, True])
def test_pingpong_with_device_policy(zero_lib, oracle_mod, staging, async_steps):
    """t, the loss scale and the current set all kept on the device, steps
    enqueued back to back; steps 3 and 4 overflow and are skipped."""
    _policy_run(zero_lib, oracle_mod, out_of_place=True, skip=True, bad_steps={3, 4}, steps=7,
                async_steps=async_steps, pingpong=True, staging=staging)


def test_pingpong_accumulation(zero_lib, oracle_mod):
    """Micro-batch accumulation with ping-pong sets: the fused last micro-batch
    reads and writes the sets the snapshot names; the skipped step 2 copies
    nothing."""
    from zero_sharded_mixed_04_gb300.optim import ZeroAdam
    dev = torch.device("cuda:0")
    N, k, psi = 4, 3, PSI_SMALL
    psi_pad = -(-psi // (N * 128)) * (N * 128)
    master = torch.zeros(psi_pad)
    master[:psi] = torch.randn(psi, generator=torch.Generator().manual_seed(17)) * 0.02
    opt = ZeroAdam(psi_pad, N, "bf16", skip_on_overflow=True, bucket_elems=131_072,
                   loss_scale=256.0, out_of_place=True, device=dev, master=master.to(dev),
                   micro_batches=k, pingpong=True)
    ref = _oracle_state(master.numpy())
    hp = oracle_mod.Hparams()
    o_t = 0
    for step in range(1, 5):
        micro = [_make_grads(N, psi, psi_pad, "bf16", 1e-3 * 256.0, 3000 * step + mb)
                 for mb in range(k)]
        if step == 2:
            micro[2][1][4321] = float("inf")
        res = opt.step_accumulated([[g.to(dev) for g in mb] for mb in micro])
        ores = oracle_mod.zero_step_accum([[_np(g) for g in mb] for mb in micro], ref["master"],
                                          ref["m"], ref["v"], ref["w"], hp, o_t + 1, 256.0, True)
        compare_result(res, ores)
        if ores["applied"]:
            o_t += 1
        assert opt.t == o_t
        compare_state(state_to_numpy(opt.state()), ref, exact=True, tag=f"step {step} ")
    assert o_t == 3 and int(opt.set_mem[0]) == 1


def test_pingpong_skip_launches_no_copy(zero_lib):
    """A skipped ping-pong step launches no restore kernel: the same number of
    kernels as an applied one, and the current-set word does not move."""
    from zero_sharded_mixed_04_gb300.optim import ZeroAdam
    Z = zero_lib
    dev = torch.device("cuda:0")
    N, n = 4, 4 * 128 * 512
    opt = ZeroAdam(n, N, "bf16", skip_on_overflow=True, out_of_place=True, device=dev,
                   loss_scale=8.0, pingpong=True)
    good = [torch.randn(n, device=dev).to(torch.bfloat16) for _ in range(N)]
    bad = [g.clone() for g in good]
    bad[2][77] = float("inf")
    launches = []
    for grads in (good, bad, good):
        before = Z.zero_launch_count()
        opt.step(grads)
        launches.append(Z.zero_launch_count() - before)
    assert launches[0] == launches[1] == launches[2]
    assert opt.t == 2 and int(opt.set_mem[0]) == 0


def _rows_area(rows):
    return 0 if rows <= 0 else 256 + rows * 2048 * 8


@pytest.mark.parametrize("rows,bucket", [(0, 400_000), (1, 400_000), (3, 400_000), (64, 400_000),
                                         (100, 16_384), (2048, 16_384)])
@pytest.mark.parametrize("clip,staging", [(0.0, 0), (0.0, 1), (0.5, 0)])
def test_norm_partials_with_few_rows(zero_lib, oracle_mod, rows, bucket, clip, staging):
    """The workspace holds `rows` rows of norm partials for a step of many
    first-pass launches (one per bucket): the launches beyond them add to the
    shared slots (each waiting for the previous launch) and the first ones
    write rows of their own.  The step, its norm and its clip must be the
    oracle's whatever the mix.  The 16K-element buckets make 184 launches,
    whose rows finalize sums over several CTAs."""
    Z = zero_lib
    dev = torch.device("cuda:0")
    N, psi = 8, PSI_MULTI_SWEEP
    psi_pad = -(-psi // (N * 128)) * (N * 128)
    launches = -(-psi_pad // bucket)
    grads = _make_grads(N, psi, psi_pad, "bf16", 1e-3 * 1024, 4242)
    master = torch.zeros(psi_pad)
    master[:psi] = torch.randn(psi, generator=torch.Generator().manual_seed(7)) * 0.02
    src = [master.to(dev), torch.zeros(psi_pad, device=dev), torch.zeros(psi_pad, device=dev),
           torch.zeros(psi_pad, dtype=torch.int16, device=dev)]
    dst = [torch.empty_like(t) for t in src]
    hp = Z.make_hparams(max_grad_norm=clip, skip_on_overflow=True, bucket_elems=bucket)
    need = Z.ZERO_WORKSPACE_CONTROL_BYTES + (4 * psi_pad if clip > 0 else 0)
    ws_bytes = need + _rows_area(rows)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    res = torch.zeros(4, dtype=torch.int32, pin_memory=True)
    plan = Z.zero_plan()
    dev_grads = [g.to(dev) for g in grads]
    assert Z.zero_plan_init(plan, dev_grads, Z.ZERO_GRAD_BF16, *src, *dst, psi_pad, N, hp, 1024.0,
                            ws, ws_bytes) == Z.ZERO_OK
    assert plan.row_capacity == rows
    plan.smem_staging = Z.ZERO_STAGING_TMA if staging else Z.ZERO_STAGING_REGISTERS
    assert Z.zero_plan_begin(plan, None) == Z.ZERO_OK
    for b0 in range(0, psi_pad, bucket):
        assert Z.zero_plan_bucket(plan, b0, min(psi_pad, b0 + bucket), None, None) == Z.ZERO_OK
    assert plan.rows_used == min(rows, launches)
    assert plan.shared_slots_used == (1 if rows < launches else 0)
    assert Z.zero_plan_end(plan, res, None) == Z.ZERO_OK
    torch.cuda.synchronize()
    ref = _oracle_state(master.numpy())
    ores = oracle_mod.zero_step([_np(g) for g in grads], ref["master"], ref["m"], ref["v"],
                                ref["w"], oracle_mod.Hparams(max_grad_norm=clip), 1, 1024.0, True)
    raw = res.clone()
    got_res = {"applied": int(raw[0]) == Z.ZERO_OK, "found_nonfinite": bool(int(raw[1])),
               "grad_norm": float(raw[2:3].view(torch.float32)[0]),
               "clip_coef": float(raw[3:4].view(torch.float32)[0])}
    compare_result(got_res, ores)
    got = {"master": dst[0].cpu().numpy(), "m": dst[1].cpu().numpy(), "v": dst[2].cpu().numpy(),
           "w": dst[3].cpu().numpy().view(np.uint16)}
    compare_state(got, ref, exact=clip == 0.0)


def test_norm_is_the_same_on_every_run(zero_lib):
    """With rows, shared slots or a mix, the norm's sum is formed in an order
    fixed by the sizes: the same step run again gives the same bits."""
    Z = zero_lib
    dev = torch.device("cuda:0")
    N, psi_pad, bucket = 4, 2_000_896, 8192
    g = torch.Generator(device="cpu").manual_seed(11)
    grads = [(torch.randn(psi_pad, generator=g) * 3e-2).to(torch.bfloat16).to(dev) for _ in range(N)]
    hp = Z.make_hparams(max_grad_norm=1.0, bucket_elems=bucket)
    need = Z.ZERO_WORKSPACE_CONTROL_BYTES + 4 * psi_pad
    norms = {}
    for rows in (0, 50, 2048):
        for rep in range(3):
            master = torch.zeros(psi_pad, device=dev)
            st = [master, torch.zeros_like(master), torch.zeros_like(master),
                  torch.zeros(psi_pad, dtype=torch.int16, device=dev)]
            ws = torch.empty(need + _rows_area(rows), dtype=torch.uint8, device=dev)
            res = torch.zeros(4, dtype=torch.int32, pin_memory=True)
            assert Z.zero_step(grads, Z.ZERO_GRAD_BF16, *st, psi_pad, N, hp, 1.0, ws, ws.numel(),
                               res) == Z.ZERO_OK
            torch.cuda.synchronize()
            norms.setdefault(rows, set()).add(int(res[2]))
    for rows, bits in norms.items():
        assert len(bits) == 1, (rows, bits)


@pytest.mark.parametrize("sigma,dtype,clip", [
    (1e25, "fp32", 1.0),    # squares overflow FP32: the norm stays finite and the clip bites
    (1e25, "fp32", 0.0),    # the norm is reported; Adam's own g*g overflows on both sides
    (3e30, "bf16", 1.0),
    (1e-30, "fp32", 0.0),   # squares underflow FP32: the norm is still reported
    (1e-30, "fp32", 1e-28),
    (1e-40, "fp32", 0.0),   # subnormal gradients: the divisions' and roots' slow paths
])
def test_norm_of_extreme_magnitudes(zero_lib, oracle_mod, sigma, dtype, clip):
    """The global norm is the square root of the exact sum of squares (the
    oracle sums FP64 squares).  Gradients whose FP32 squares would overflow or
    underflow must give the oracle's norm and clip coefficient all the same."""
    run_parity(zero_lib, oracle_mod, N=4, psi=PSI_SMALL, dtype=dtype, steps=2, clip=clip,
               sigma=sigma, loss_scale=1.0)
