"""GPU parity on the five benchmark workloads at their full sizes.

flat1m_n4 and gpt2small_n4 are compared with the oracle over the whole
vector, every step.  The three large workloads do not fit the host.  For
each step the oracle reads every rank's gradient from the device once, in
chunks on host threads, to form the step-wide overflow flag and norm itself.
It then steps sampled windows of 2^20 elements:
  - the first and last elements of every owner's slice;
  - the ragged tail and the padding;
  - the 2^31 and 2^32 element boundaries;
  - bucket edges and the injected +inf;
  - the boundaries between the launches a bucket (or the whole vector) is
    split into;
  - 64 seeded random windows.
It compares each window with the device state, element by element.
"""
from __future__ import annotations

import concurrent.futures
import gc
import math
import os

import numpy as np
import pytest
import torch

from parity_util import compare_result, compare_state, state_to_numpy

pytestmark = pytest.mark.gpu

WIN = 1 << 20
N_RANDOM = 64
CHUNK = 1 << 24
THREADS = max(1, min(16, os.cpu_count() or 1))


def _free():
    gc.collect()
    torch.cuda.empty_cache()


def _launch_splits(b0, b1):
    """Where the library splits the range [b0, b1) of one pass into kernel
    launches: near-equal parts of at most 2^22 elements, each part a multiple
    of 256 elements except the last."""
    groups = (b1 - b0) // 8
    parts = -(-(groups * 8) // (1 << 22))
    per = -(-groups // parts)
    per = -(-per // 32) * 32
    return [b0 + k * per * 8 for k in range(1, parts) if k * per < groups]


def _windows(wl, psi_pad, shard, extra=(), n_random=N_RANDOM, seed=0):
    wins = []
    for r in range(wl.N):
        wins += [(r * shard, r * shard + WIN), ((r + 1) * shard - WIN, (r + 1) * shard)]
    wins.append((wl.psi - WIN, psi_pad))
    for edge in (1 << 31, 1 << 32):
        if edge + WIN < psi_pad:
            wins.append((edge - WIN, edge + WIN))     # 2^31 +- 2^20 and 2^32 +- 2^20
    splits = []
    if wl.bucket_elems:
        for k in (1, 2, 17, psi_pad // wl.bucket_elems):
            e = k * wl.bucket_elems
            if WIN < e < psi_pad - WIN:
                wins.append((e - WIN // 2, e + WIN // 2))
        # every launch boundary inside the first bucket and one in the middle
        for k in (0, 17):
            b0 = k * wl.bucket_elems
            splits += _launch_splits(b0, min(psi_pad, b0 + wl.bucket_elems))
    else:
        cuts = _launch_splits(0, psi_pad)
        near = [c for c in cuts for edge in (1 << 31, 1 << 32) if abs(c - edge) < (1 << 22)]
        splits += cuts[:3] + near + cuts[-2:]
    for c in splits:
        wins.append((c - WIN // 2, c + WIN // 2))
    for c in extra:
        wins.append((max(0, c - WIN // 2), min(psi_pad, c + WIN // 2)))
    rng = np.random.Generator(np.random.Philox(seed))
    for _ in range(n_random):
        lo = int(rng.integers(0, psi_pad - WIN))
        wins.append((lo, lo + WIN))
    # clamp, align to 8 elements and merge overlaps
    wins = sorted((max(0, lo) // 8 * 8, min(psi_pad, -(-hi // 8) * 8)) for lo, hi in wins)
    merged = []
    for lo, hi in wins:
        if merged and lo <= merged[-1][1]:
            merged[-1] = (merged[-1][0], max(merged[-1][1], hi))
        else:
            merged.append((lo, hi))
    return merged


def _grad_np(t: torch.Tensor) -> np.ndarray:
    from zero_sharded_mixed_04_gb300 import synth
    return synth.to_numpy_grad(t)


def _oracle_check(oracle_mod, grads, N, scale, psi_pad):
    """The oracle's step-wide overflow flag and sum of squares over the whole
    vector.  Chunks run on host threads (the oracle releases the GIL).  The
    chunk sums are combined in flat order, so only the FP64 rounding order
    differs from one sequential pass."""
    def one(c0):
        acc = oracle_mod.CheckAccumulator(N, scale)
        acc.feed([_grad_np(g[c0:c0 + CHUNK]) for g in grads])
        return acc.found_nonfinite, acc.sumsq
    with concurrent.futures.ThreadPoolExecutor(THREADS) as ex:
        parts = list(ex.map(one, range(0, psi_pad, CHUNK)))
    return any(p[0] for p in parts), math.fsum(p[1] for p in parts)


def _run_workload(zero_lib, oracle_mod, name, out_of_place, full_compare, steps=None,
                  device_policy=False, staging=0, pingpong=False):
    from zero_sharded_mixed_04_gb300 import synth
    from zero_sharded_mixed_04_gb300.optim import ZeroAdam
    wl = synth.WORKLOADS[name]
    dev = torch.device("cuda:0")
    steps = steps or wl.steps
    psi_pad, N = wl.psi_pad, wl.N
    shard = psi_pad // N
    master = synth.make_master(wl, dev)
    opt = ZeroAdam(psi_pad, N, wl.grad_dtype, lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2,
                   eps=wl.eps, weight_decay=wl.weight_decay, max_grad_norm=wl.max_grad_norm,
                   skip_on_overflow=wl.skip_on_overflow, bucket_elems=wl.bucket_elems,
                   loss_scale=wl.loss_scale, dynamic_loss_scale=wl.dynamic_loss_scale,
                   out_of_place=out_of_place, device=dev, master=master,
                   device_policy=device_policy, smem_staging=staging, pingpong=pingpong)
    del master
    _free()
    hp = oracle_mod.Hparams(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps,
                            weight_decay=wl.weight_decay, max_grad_norm=wl.max_grad_norm)
    extra = []
    if wl.inject_inf_step:
        extra.append(synth.inf_index(wl, wl.inject_inf_step)[1])
    wins = [(0, psi_pad)] if full_compare else _windows(wl, psi_pad, shard, extra, seed=wl.index)
    ref = {w: state_to_numpy(opt.state(), *w) for w in wins}
    grads = None
    o_t, o_scale, o_good = 0, wl.loss_scale, 0
    exact = wl.max_grad_norm == 0.0
    for step in range(1, steps + 1):
        grads = synth.make_grads(wl, step, dev, loss_scale=o_scale, out=grads)
        gw = {w: [_grad_np(g[w[0]:w[1]]) for g in grads] for w in wins}
        # the oracle's own pass over the whole gradient
        if full_compare:
            acc = oracle_mod.CheckAccumulator(N, o_scale)
            acc.feed(gw[wins[0]])
            found, sumsq = acc.found_nonfinite, acc.sumsq
        else:
            found, sumsq = _oracle_check(oracle_mod, grads, N, o_scale, psi_pad)
        res = opt.step(grads)
        applied = not (wl.skip_on_overflow and found)
        coef = (oracle_mod.clip_coef_from_sumsq(wl.max_grad_norm, sumsq)
                if wl.max_grad_norm > 0 and applied else None)
        ores = {"applied": applied, "found_nonfinite": found,
                "grad_norm": float(np.float32(math.sqrt(sumsq))),
                "clip_coef": 1.0 if coef is None else coef}
        compare_result(res, ores)
        if wl.inject_inf_step:
            assert res["applied"] == (step != wl.inject_inf_step)
        def step_one(w):
            r = ref[w]
            oracle_mod.step_window(gw[w], r["master"], r["m"], r["v"], r["w"], hp, o_t + 1,
                                   o_scale, applied, coef)
        with concurrent.futures.ThreadPoolExecutor(THREADS) as ex:
            list(ex.map(step_one, wins))
        for w in wins:
            compare_state(state_to_numpy(opt.state(), *w), ref[w], exact, offset=w[0],
                          tag=f"{name} step {step} ")
        if applied:
            o_t += 1
        if wl.dynamic_loss_scale:
            o_scale, o_good = oracle_mod.loss_scale_update(o_scale, o_good, found, 2000, 0.5,
                                                           2.0)
        assert opt.t == o_t and opt.scaler.scale == o_scale
        del gw
    del grads, opt
    _free()


def test_flat1m_n4(zero_lib, oracle_mod):
    _run_workload(zero_lib, oracle_mod, "flat1m_n4", out_of_place=False, full_compare=True)


def test_gpt2small_n4(zero_lib, oracle_mod):
    _run_workload(zero_lib, oracle_mod, "gpt2small_n4", out_of_place=False, full_compare=True)


@pytest.mark.parametrize("out_of_place", [True, False])
def test_flat1b_n8(zero_lib, oracle_mod, out_of_place):
    _run_workload(zero_lib, oracle_mod, "flat1b_n8", out_of_place=out_of_place,
                  full_compare=False)


def test_flat3b_n4_fp32(zero_lib, oracle_mod):
    _run_workload(zero_lib, oracle_mod, "flat3b_n4_fp32", out_of_place=False, full_compare=False)


def test_ragged6b_n4(zero_lib, oracle_mod):
    _run_workload(zero_lib, oracle_mod, "ragged6b_n4", out_of_place=False, full_compare=False)


def test_ragged6b_n4_staged(zero_lib, oracle_mod):
    """The TMA-staged one-pass kernel past the 2^31 and 2^32 element
    boundaries (6e9 parameters)."""
    _run_workload(zero_lib, oracle_mod, "ragged6b_n4", out_of_place=False, full_compare=False,
                  staging=zero_lib.ZERO_STAGING_TMA)


def test_gpt2small_n4_staged(zero_lib, oracle_mod):
    _run_workload(zero_lib, oracle_mod, "gpt2small_n4", out_of_place=False, full_compare=True,
                  staging=zero_lib.ZERO_STAGING_TMA)


def test_flat1b_n8_as_benchmarked(zero_lib, oracle_mod):
    """The path bench.py times: out of place with ping-pong state sets, through
    the plan entry points, with t and the loss scale kept on the device and
    every tile staged in shared memory by TMA; the injected +inf on step 3
    must be skipped (the current set stays current) and halve the scale."""
    _run_workload(zero_lib, oracle_mod, "flat1b_n8", out_of_place=True, full_compare=False,
                  device_policy=True, staging=zero_lib.ZERO_STAGING_TMA, pingpong=True)


def test_flat1b_n8_staged_with_restore_copy(zero_lib, oracle_mod):
    """The same without ping-pong sets: a skipped step copies src into dst."""
    _run_workload(zero_lib, oracle_mod, "flat1b_n8", out_of_place=True, full_compare=False,
                  device_policy=True, staging=zero_lib.ZERO_STAGING_TMA)


def test_flat1b_n8_register_kernel_with_device_policy(zero_lib, oracle_mod):
    """bench.py --staging registers: the same path with the register kernel."""
    _run_workload(zero_lib, oracle_mod, "flat1b_n8", out_of_place=True, full_compare=False,
                  device_policy=True, pingpong=True)
