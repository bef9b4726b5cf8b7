"""Pins of the oracle's step-wide decisions: overflow skip, global-norm clip,
dynamic loss scale, and the windowed form used for vectors too large for the
host."""
import math

import numpy as np
import pytest
import torch


def _setup(rng, N, psi_pad, psi, dtype="bf16", sigma=1e-3, oracle_mod=None):
    grads = []
    for _ in range(N):
        g = np.zeros(psi_pad, np.float32)
        g[:psi] = rng.standard_normal(psi) * sigma
        grads.append(oracle_mod.f32_to_bf16(g) if dtype == "bf16" else g)
    master = np.zeros(psi_pad, np.float32)
    master[:psi] = rng.standard_normal(psi) * 0.02
    return grads, master, np.zeros(psi_pad, np.float32), np.zeros(psi_pad, np.float32), \
        oracle_mod.f32_to_bf16(master)


@pytest.mark.parametrize("bad", [np.inf, -np.inf, np.nan])
def test_skip_leaves_state_bit_unchanged(oracle_mod, bad):
    rng = np.random.default_rng(5)
    N, psi_pad = 4, 4 * 128 * 2
    grads, master, m, v, w = _setup(rng, N, psi_pad, psi_pad - 9, oracle_mod=oracle_mod)
    hp = oracle_mod.Hparams()
    oracle_mod.zero_step(grads, master, m, v, w, hp, 1)  # one applied step first
    before = [a.copy() for a in (master, m, v, w)]
    grads[1] = grads[1].copy()
    grads[1][77] = oracle_mod.f32_to_bf16(np.array([bad], np.float32))[0]
    res = oracle_mod.zero_step(grads, master, m, v, w, hp, 2, 65536.0, skip_on_overflow=True)
    assert res["found_nonfinite"] and not res["applied"]
    for a, b in zip((master, m, v, w), before):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    # without the skip the non-finite value flows into the state
    res = oracle_mod.zero_step(grads, master, m, v, w, hp, 2, 65536.0, skip_on_overflow=False)
    assert res["found_nonfinite"] and res["applied"]
    assert not np.isfinite(master[77])


def test_fp32_sum_overflow_is_detected(oracle_mod):
    """Two finite BF16 contributions near the top of the range overflow the
    FP32 sum; the check sits on the reduced gradient, so it sees that."""
    N, psi_pad = 2, 256
    big = oracle_mod.f32_to_bf16(np.full(psi_pad, 3.0e38, np.float32))
    assert np.isfinite(oracle_mod.bf16_to_f32(big)).all()
    master = np.zeros(psi_pad, np.float32)
    m, v, w = np.zeros_like(master), np.zeros_like(master), np.zeros(psi_pad, np.uint16)
    res = oracle_mod.zero_step([big, big], master, m, v, w, oracle_mod.Hparams(), 1,
                               1.0, skip_on_overflow=True)
    assert res["found_nonfinite"] and not res["applied"]


@pytest.mark.parametrize("max_norm,sigma", [(1.0, 1e-3), (0.01, 1e-3), (1e-4, 1e-2)])
def test_clip_matches_torch(oracle_mod, max_norm, sigma):
    """N = 1: clip_grad_norm_ followed by one Adam step, in torch on the CPU."""
    rng = np.random.default_rng(9)
    n = 128 * 64
    g = (rng.standard_normal(n) * sigma).astype(np.float32)
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    master, m, v, w = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32), \
        np.zeros(n, np.uint16)
    hp = oracle_mod.Hparams(max_grad_norm=max_norm)
    res = oracle_mod.zero_step([g.copy()], master, m, v, w, hp, 1)
    tp = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    tp.grad = torch.from_numpy(g.astype(np.float64).astype(np.float32))
    tp64 = torch.from_numpy(g.astype(np.float64))
    norm = torch.nn.utils.clip_grad_norm_([tp], max_norm)
    assert math.isclose(res["grad_norm"], float(torch.linalg.vector_norm(tp64)), rel_tol=1e-7)
    assert math.isclose(res["grad_norm"], float(norm), rel_tol=1e-6)
    coef = min(1.0, max_norm / (float(torch.linalg.vector_norm(tp64)) + 1e-6))
    assert math.isclose(res["clip_coef"], coef, rel_tol=1e-7)
    opt = torch.optim.Adam([tp], lr=hp.lr, betas=(hp.beta1, hp.beta2), eps=hp.eps,
                           foreach=False, fused=False)
    opt.step()
    rms_m = float(np.sqrt(np.mean(m.astype(np.float64) ** 2)))
    assert np.max(np.abs(m - opt.state[tp]["exp_avg"].numpy())) <= 2e-6 * rms_m
    rms_p = float(np.sqrt(np.mean(master.astype(np.float64) ** 2)))
    assert np.max(np.abs(master - tp.detach().numpy())) <= 1e-6 * rms_p


def test_clip_norm_is_global_over_all_owners(oracle_mod):
    """The clip coefficient comes from the norm over every owner's slice:
    clipping never triggers from one shard alone."""
    rng = np.random.default_rng(2)
    N, psi_pad = 4, 4 * 128
    grads, master, m, v, w = _setup(rng, N, psi_pad, psi_pad, "fp32", sigma=1.0,
                                    oracle_mod=oracle_mod)
    full = oracle_mod.all_reduce(grads, psi_pad, np.float32(1.0 / N)).astype(np.float64)
    hp = oracle_mod.Hparams(max_grad_norm=1.0)
    res = oracle_mod.zero_step(grads, master, m, v, w, hp, 1)
    assert math.isclose(res["grad_norm"], float(np.linalg.norm(full)), rel_tol=1e-7)
    shard_norm = float(np.linalg.norm(full[:psi_pad // N]))
    assert res["grad_norm"] > shard_norm
    assert math.isclose(res["clip_coef"], 1.0 / (float(np.linalg.norm(full)) + 1e-6), rel_tol=1e-7)


def test_loss_scale_matches_torch_amp_update(oracle_mod):
    """The dynamic loss scale against torch's own scale-update routine."""
    flags = [0, 0, 1, 0, 0, 0, 0, 1, 1, 0, 0, 0, 0, 0, 0, 0]
    interval = 3
    scale, good = 65536.0, 0
    t_scale = torch.tensor([65536.0])
    t_track = torch.tensor([0], dtype=torch.int32)
    for f in flags:
        scale, good = oracle_mod.loss_scale_update(scale, good, bool(f), interval, 0.5, 2.0)
        torch._amp_update_scale_(t_scale, t_track, torch.tensor([float(f)]), 2.0, 0.5, interval)
        assert scale == float(t_scale) and good == int(t_track)


@pytest.mark.parametrize("clip", [0.0, 0.5])
def test_windowed_form_equals_whole_step(oracle_mod, clip):
    rng = np.random.default_rng(21)
    N, psi_pad, psi = 4, 4 * 128 * 5, 4 * 128 * 5 - 200
    grads, master, m, v, w = _setup(rng, N, psi_pad, psi, "bf16", sigma=1e-3 * 8,
                                    oracle_mod=oracle_mod)
    hp = oracle_mod.Hparams(max_grad_norm=clip, weight_decay=0.1)
    whole = [a.copy() for a in (master, m, v, w)]
    res = oracle_mod.zero_step(grads, *whole, hp, 1, 8.0)
    acc = oracle_mod.CheckAccumulator(N, 8.0)
    for s in range(0, psi_pad, 700):
        acc.feed([g[s:s + 700] for g in grads])
    assert acc.found_nonfinite == res["found_nonfinite"]
    assert acc.sumsq == res["sumsq"]
    coef = oracle_mod.clip_coef_from_sumsq(clip, acc.sumsq) if clip else None
    if clip:
        assert coef == res["clip_coef"]
    for s in range(0, psi_pad, 300):
        win = slice(s, min(psi_pad, s + 300))
        parts = [np.ascontiguousarray(a[win]) for a in (master, m, v, w)]
        oracle_mod.step_window([np.ascontiguousarray(g[win]) for g in grads], *parts, hp, 1, 8.0,
                               True, coef)
        for a, p in zip((master, m, v, w), parts):
            a[win] = p
    for a, b in zip((master, m, v, w), whole):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


@pytest.mark.parametrize("c", [1e30, 1e25, 3e19, 1.0, 1e-20, 1e-30, 1e-40])
def test_norm_is_the_closed_form_at_any_magnitude(oracle_mod, c):
    """Every rank sends the same FP32 gradient c, so the batch-mean gradient is
    c in every one of the n elements, to within the rounding of the FP32 rank
    sum (N = 4, loss scale 1), and its norm is |c| * sqrt(n).  That holds where c*c overflows FP32 (c >= 2^64)
    or underflows it (c < 2^-75): the norm is the square root of the sum of
    squares, not of a sum that saturated."""
    N, n = 4, 4 * 128 * 8
    g = np.full(n, c, np.float32)
    cf = float(np.float32(c))            # the value FP32 holds (1e-40 is subnormal)
    master = np.zeros(n, np.float32)
    m, v, w = np.zeros_like(master), np.zeros_like(master), np.zeros(n, np.uint16)
    res = oracle_mod.zero_step([g] * N, master, m, v, w, oracle_mod.Hparams(), 1, 1.0)
    want = abs(cf) * math.sqrt(n)
    assert res["grad_norm"] == pytest.approx(want, rel=1e-6)
    # with a clip bound the coefficient follows from that norm
    master = np.zeros(n, np.float32)
    m, v, w = np.zeros_like(master), np.zeros_like(master), np.zeros(n, np.uint16)
    res = oracle_mod.zero_step([g] * N, master, m, v, w, oracle_mod.Hparams(max_grad_norm=1.0), 1,
                               1.0)
    assert res["clip_coef"] == pytest.approx(min(1.0, 1.0 / (want + 1e-6)), rel=1e-6)
