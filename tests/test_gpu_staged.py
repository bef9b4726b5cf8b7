"""GPU parity of the shared-memory-staged one-pass kernel (ZERO_STAGING_TMA).

Each 2048-element tile is copied into a shared-memory stage by TMA bulk copies
and computed from there.  The results must equal the oracle's bit for bit, as
the register kernel's do.  Sizes give ragged last tiles and several tiles per
CTA.  The cases cover the rank counts, both gradient types, in place and out
of place, skips, buckets, split sub-launches, gradients staged through device
slots, the device policy, and the bounded waits running out.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from parity_util import compare_result, compare_state, state_to_numpy
from test_gpu_parity import (PSI_MULTI_SWEEP, PSI_SMALL, _make_grads, _np, _oracle_state,
                             run_parity)

pytestmark = pytest.mark.gpu

TMA = 1  # ZERO_STAGING_TMA


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_staged_one_pass_in_place(zero_lib, oracle_mod, N, dtype):
    psi = PSI_MULTI_SWEEP if N in (4, 8) else PSI_SMALL
    run_parity(zero_lib, oracle_mod, N=N, psi=psi, dtype=dtype, staging=TMA)


@pytest.mark.parametrize("N,dtype,psi", [(8, "bf16", PSI_MULTI_SWEEP), (4, "fp32", PSI_SMALL),
                                         (5, "bf16", PSI_SMALL)])
def test_staged_skip_out_of_place(zero_lib, oracle_mod, N, dtype, psi):
    """Step 2 carries a +inf and is skipped: the staged kernel has written dst,
    and the restore puts src back."""
    run_parity(zero_lib, oracle_mod, N=N, psi=psi, dtype=dtype, steps=4, skip=True,
               out_of_place=True, bad_step=2, loss_scale=1024.0, dynamic=True, staging=TMA)


def test_staged_weight_decay_and_buckets(zero_lib, oracle_mod):
    run_parity(zero_lib, oracle_mod, N=4, psi=PSI_MULTI_SWEEP, wd=0.1, bucket=400_000, steps=3,
               staging=TMA, api="plan")


def test_staged_split_sub_launches(zero_lib, oracle_mod):
    """One bucket of 9M elements: the library splits it into sub-launches of
    at most 4M elements, chained by programmatic dependent launch."""
    run_parity(zero_lib, oracle_mod, N=2, psi=9_000_001, steps=2, out_of_place=True,
               skip=True, staging=TMA)


def test_staged_with_device_policy(zero_lib, oracle_mod):
    """The benchmark's form: out of place, skip on overflow, t and the dynamic
    loss scale kept on the device."""
    run_parity(zero_lib, oracle_mod, N=8, psi=PSI_MULTI_SWEEP, steps=4, skip=True,
               out_of_place=True, bad_step=3, loss_scale=4096.0, dynamic=True,
               growth_interval=2, bucket=1_000_000, staging=TMA, device_policy=True)


def test_staged_from_host_slots(zero_lib, oracle_mod):
    """Gradients in pinned host memory stream through two device slots: each
    bucket's copies start at the slot's base (a bucket offset), not at the
    gradient vector's."""
    from zero_sharded_mixed_04_gb300.optim import ZeroAdam
    dev = torch.device("cuda:0")
    N, psi, bucket = 4, PSI_MULTI_SWEEP, 262_144
    psi_pad = -(-psi // (N * 128)) * (N * 128)
    master = torch.zeros(psi_pad)
    master[:psi] = torch.randn(psi, generator=torch.Generator().manual_seed(31)) * 0.02
    opt = ZeroAdam(psi_pad, N, "bf16", bucket_elems=bucket, out_of_place=True, device=dev,
                   master=master.to(dev), smem_staging=TMA)
    slots = opt.make_slots()
    copy_stream = torch.cuda.Stream(dev)
    ref = _oracle_state(master.numpy())
    hp = oracle_mod.Hparams()
    for step in (1, 2):
        grads = _make_grads(N, psi, psi_pad, "bf16", 1e-3, 555 + step)
        host = [g.pin_memory() for g in grads]
        opt.enqueue_from_host(host, slots, copy_stream)
        res = opt.finish()
        ores = oracle_mod.zero_step([_np(g) for g in grads], ref["master"], ref["m"], ref["v"],
                                    ref["w"], hp, step, 1.0, False)
        compare_result(res, ores)
        compare_state(state_to_numpy(opt.state()), ref, exact=True, tag=f"step {step} ")


def _plan_step(Z, grads, src, dst, n, N, hp, staging, res):
    ws = torch.empty(Z.zero_workspace_bytes(n, hp, src[0].data_ptr() == dst[0].data_ptr()),
                     dtype=torch.uint8, device=grads[0].device)
    plan = Z.zero_plan()
    assert Z.zero_plan_init(plan, grads, Z.ZERO_GRAD_BF16, *src, *dst, n, N, hp, 1.0, ws,
                            ws.numel()) == Z.ZERO_OK
    plan.smem_staging = staging
    assert Z.zero_plan_begin(plan, None) == Z.ZERO_OK
    assert Z.zero_plan_bucket(plan, 0, n, None, None) == Z.ZERO_OK
    assert Z.zero_plan_end(plan, res, None) == Z.ZERO_OK
    torch.cuda.synchronize()
    return int(res[0])


@pytest.mark.parametrize("n", [32_768, 4_194_304])
def test_staged_wait_runs_out(zero_lib, n):
    """CTA 0 never copies its first tile (ZERO_STAGING_TMA_TEST_STALL), so its
    consumers' wait runs out after about a second.  With more tiles per CTA
    than stages (the larger case: 2048 tiles of 2048 elements over at most 304
    CTAs), the producer's wait for a free stage runs out too, and it then
    waits for the copies it issued.  The step ends with ZERO_ERR_TIMEOUT and,
    out of place, leaves dst equal to src.  The context stays usable: the next
    step, staged, equals the register kernel's bit for bit."""
    Z = zero_lib
    dev = torch.device("cuda:0")
    N = 4
    grads = [(torch.randn(n, generator=torch.Generator().manual_seed(60 + i)) * 1e-3).to(
        torch.bfloat16).to(dev) for i in range(N)]
    src = [torch.randn(n, device=dev) * 0.02, torch.rand(n, device=dev) * 1e-4,
           torch.rand(n, device=dev) * 1e-6, torch.zeros(n, dtype=torch.int16, device=dev)]
    before = [t.clone() for t in src]
    dst = [torch.full_like(t, 7) for t in src]
    hp = Z.make_hparams(step=3)
    res = torch.zeros(4, dtype=torch.int32, pin_memory=True)
    assert _plan_step(Z, grads, src, dst, n, N, hp, Z.ZERO_STAGING_TMA_TEST_STALL,
                      res) == Z.ZERO_ERR_TIMEOUT
    for a, b in zip(dst, before):
        assert torch.equal(a, b)
    for a, b in zip(src, before):
        assert torch.equal(a, b)
    # the context still works, and both forms agree
    assert _plan_step(Z, grads, src, dst, n, N, hp, Z.ZERO_STAGING_TMA, res) == Z.ZERO_OK
    dst_reg = [torch.full_like(t, 7) for t in src]
    assert _plan_step(Z, grads, src, dst_reg, n, N, hp, Z.ZERO_STAGING_REGISTERS,
                      res) == Z.ZERO_OK
    for a, b in zip(dst, dst_reg):
        assert torch.equal(a, b)
    assert not torch.equal(dst[0], before[0])


def test_staged_rejects_stages_that_do_not_fit(zero_lib):
    """Two stages for N = 64 FP32 gradients would need 1.1 MB: the plan
    refuses before launching anything."""
    Z = zero_lib
    dev = torch.device("cuda:0")
    N, n = 64, 64 * 128
    grads = [torch.zeros(n, device=dev) for _ in range(N)]
    st = [torch.zeros(n, device=dev) for _ in range(3)] + [torch.zeros(n, dtype=torch.int16,
                                                                       device=dev)]
    hp = Z.make_hparams()
    ws = torch.empty(Z.zero_workspace_bytes(n, hp, True), dtype=torch.uint8, device=dev)
    plan = Z.zero_plan()
    assert Z.zero_plan_init(plan, grads, Z.ZERO_GRAD_FP32, *st, *st, n, N, hp, 1.0, ws,
                            ws.numel()) == Z.ZERO_OK
    plan.smem_staging = Z.ZERO_STAGING_TMA
    assert Z.zero_plan_begin(plan, None) == Z.ZERO_OK
    assert Z.zero_plan_bucket(plan, 0, n, None, None) == Z.ZERO_ERR_ARG
    plan.smem_staging = 5
    assert Z.zero_plan_bucket(plan, 0, n, None, None) == Z.ZERO_ERR_ARG


def test_staged_rejects_host_gradients(zero_lib):
    """TMA copies read device memory only: gradients in pinned host memory are
    refused (the register kernel may read them)."""
    Z = zero_lib
    dev = torch.device("cuda:0")
    N, n = 2, 2 * 128 * 8
    grads = [torch.zeros(n, dtype=torch.bfloat16).pin_memory() for _ in range(N)]
    st = [torch.zeros(n, device=dev) for _ in range(3)] + [torch.zeros(n, dtype=torch.int16,
                                                                       device=dev)]
    hp = Z.make_hparams()
    ws = torch.empty(Z.zero_workspace_bytes(n, hp, True), dtype=torch.uint8, device=dev)
    plan = Z.zero_plan()
    assert Z.zero_plan_init(plan, grads, Z.ZERO_GRAD_BF16, *st, *st, n, N, hp, 1.0, ws,
                            ws.numel()) == Z.ZERO_OK
    plan.smem_staging = Z.ZERO_STAGING_TMA
    assert Z.zero_plan_begin(plan, None) == Z.ZERO_OK
    assert Z.zero_plan_bucket(plan, 0, n, None, None) == Z.ZERO_ERR_ARG


@pytest.mark.parametrize("psi", [1, 7, 1023, 2049])
def test_staged_tiny_vectors(zero_lib, oracle_mod, psi):
    """A single partial tile (one to a few hundred 8-element groups), out of
    place with the skip on and in place without it."""
    run_parity(zero_lib, oracle_mod, N=4, psi=psi, steps=2, staging=TMA)
    run_parity(zero_lib, oracle_mod, N=8, psi=psi, steps=3, skip=True, out_of_place=True,
               bad_step=2, staging=TMA)


def test_staged_empty_plan(zero_lib):
    """An empty vector through the plan with staging: no bucket, the step
    completes and reports success."""
    Z = zero_lib
    hp = Z.make_hparams(skip_on_overflow=True)
    ws = torch.empty(Z.zero_workspace_bytes(0, hp, False), dtype=torch.uint8, device="cuda")
    plan = Z.zero_plan()
    assert Z.zero_plan_init(plan, [None, None], Z.ZERO_GRAD_BF16, None, None, None, None, None,
                            None, None, None, 0, 2, hp, 1.0, ws, ws.numel()) == Z.ZERO_OK
    plan.smem_staging = Z.ZERO_STAGING_TMA
    assert Z.zero_plan_begin(plan, None) == Z.ZERO_OK
    assert Z.zero_plan_end(plan, None, None) == Z.ZERO_OK
