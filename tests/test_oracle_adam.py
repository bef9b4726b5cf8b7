"""Pins of the oracle's owner update (mixed-precision Adam/AdamW).

* N = 1 with loss scale 1 reduces the step to one optimizer step on one
  gradient: it must agree with torch.optim.Adam/AdamW on the CPU in FP32 (a
  library routine) to FP32 rounding noise.
* Closed forms: from m = v = 0 the first step moves every weight by
  -lr * g / (|g| + eps); a constant gradient keeps moving it by that amount;
  with zero gradient AdamW only decays the weight by (1 - lr*wd) per step.
"""
import math

import numpy as np
import pytest
import torch


def _bf16_grad(oracle_mod, rng, n, sigma):
    return oracle_mod.f32_to_bf16((rng.standard_normal(n) * sigma).astype(np.float32))


def _state(n, p0):
    return p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)


def _scale_close(a, b, tol):
    """|a - b| <= tol * rms(b): error measured against the array's scale, so
    that values passing through zero (cancellation) do not dominate."""
    rms = math.sqrt(float(np.mean(np.asarray(b, np.float64) ** 2))) or 1.0
    err = float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64))))
    assert err <= tol * rms, f"max err {err:.3e} > {tol:.1e} * rms {rms:.3e}"


@pytest.mark.parametrize("wd", [0.0, 0.1])
@pytest.mark.parametrize("grad", ["bf16", "fp32"])
def test_n1_matches_torch_adamw(oracle_mod, wd, grad):
    rng = np.random.default_rng(7)
    n = 128 * 96
    hp = oracle_mod.Hparams(lr=1e-3, weight_decay=wd)
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    master, m, v, w = _state(n, p0)
    tp = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    cls = torch.optim.AdamW if wd else torch.optim.Adam
    opt = cls([tp], lr=hp.lr, betas=(hp.beta1, hp.beta2), eps=hp.eps, weight_decay=wd,
              foreach=False, fused=False)
    for t in range(1, 13):
        if grad == "bf16":
            gb = _bf16_grad(oracle_mod, rng, n, 1e-3)
            g32 = oracle_mod.bf16_to_f32(gb).copy()
        else:
            gb = (rng.standard_normal(n) * 1e-3).astype(np.float32)
            g32 = gb.copy()
        res = oracle_mod.zero_step([gb], master, m, v, w, hp, t)
        assert res["applied"] and not res["found_nonfinite"]
        tp.grad = torch.from_numpy(g32)
        opt.step()
    st = opt.state[tp]
    _scale_close(master, tp.detach().numpy(), 1e-6)
    _scale_close(m, st["exp_avg"].numpy(), 2e-6)
    _scale_close(v, st["exp_avg_sq"].numpy(), 2e-6)
    # the working weights are the BF16 rounding of the master weights
    assert np.array_equal(w, oracle_mod.f32_to_bf16(master))


def test_first_step_closed_form(oracle_mod):
    """t = 1 from m = v = 0: m_hat = g and v_hat = g^2, so the update is
    -lr * g / (|g| + eps); this pins both bias corrections and where eps sits."""
    g = np.concatenate([np.logspace(-12, 0, 64), -np.logspace(-12, 0, 64)]).astype(np.float32)
    n = g.size
    hp = oracle_mod.Hparams(lr=1e-3)
    master, m, v, w = _state(n, np.zeros(n, np.float32))
    oracle_mod.zero_step([g.copy()], master, m, v, w, hp, 1)
    g64 = g.astype(np.float64)
    expected = -hp.lr * g64 / (np.abs(g64) + hp.eps)
    np.testing.assert_allclose(master, expected, rtol=1e-6, atol=0)
    np.testing.assert_allclose(m, (1 - hp.beta1) * g64, rtol=1e-6, atol=0)
    np.testing.assert_allclose(v, (1 - hp.beta2) * g64 * g64, rtol=1e-6, atol=0)
    # the weight moves against the gradient
    assert (np.sign(master) == -np.sign(g)).all()


def test_constant_gradient_closed_form(oracle_mod):
    """A constant g for k steps: m_k = (1 - b1^k) g and v_k = (1 - b2^k) g^2, so
    the bias-corrected update stays -lr * g / (|g| + eps) every step."""
    g = np.array([3e-4, -2e-3, 1e-6, -0.5] * 32, dtype=np.float32)
    n = g.size
    hp = oracle_mod.Hparams(lr=1e-3)
    master, m, v, w = _state(n, np.zeros(n, np.float32))
    g64 = g.astype(np.float64)
    for k in range(1, 9):
        oracle_mod.zero_step([g.copy()], master, m, v, w, hp, k)
        np.testing.assert_allclose(m, (1 - hp.beta1 ** k) * g64, rtol=4e-6)
        np.testing.assert_allclose(v, (1 - hp.beta2 ** k) * g64 * g64, rtol=4e-6)
        np.testing.assert_allclose(master, -k * hp.lr * g64 / (np.abs(g64) + hp.eps), rtol=4e-6)


def test_decoupled_weight_decay_closed_form(oracle_mod):
    """With zero gradient the moments stay zero, the Adam term is 0/(0+eps) = 0,
    and AdamW only multiplies the weight by (1 - lr*wd) each step."""
    n = 256
    rng = np.random.default_rng(3)
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    hp = oracle_mod.Hparams(lr=1e-3, weight_decay=0.1)
    master, m, v, w = _state(n, p0)
    zero = np.zeros(n, np.float32)
    for k in range(1, 6):
        oracle_mod.zero_step([zero], master, m, v, w, hp, k)
        np.testing.assert_allclose(master, p0.astype(np.float64) * (1 - hp.lr * 0.1) ** k,
                                   rtol=2e-7 * k + 1e-7)
    assert not m.any() and not v.any()


def test_step_scalars(oracle_mod):
    hp = oracle_mod.Hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)
    for t in (1, 2, 10, 1000):
        s = oracle_mod.step_scalars(hp, t, 4, 65536.0)
        assert s["inv"] == np.float32(1.0 / (4 * 65536.0))
        assert s["step_size"] == np.float32(1e-3 / (1 - 0.9 ** t))
        assert s["sbc2"] == np.float32(math.sqrt(1 - 0.999 ** t))
        assert s["decay"] == np.float32(1 - 1e-3 * 0.1)
        assert s["omb1"] == np.float32(0.1) and s["omb2"] == np.float32(1 - 0.999)
