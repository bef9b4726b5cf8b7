"""Pins of the oracle's gradient accumulation over micro-batches.

* k = 1 is the plain step, bit for bit.
* Integer-valued gradients make every partial sum exact.  A step on k
  micro-batches then equals one plain step on the per-rank integer sums with
  the loss scale multiplied by k, bit for bit.
* N = 1 against torch: accumulate the micro-batch gradients divided by k
  into .grad, then take one Adam step (a library routine), within FP32
  rounding noise.
* A non-finite value in any micro-batch makes the accumulated gradient
  non-finite, so the step is skipped.
* Hand-worked FP32 cases whose bits depend on the micro-batches being added
  in order, to an accumulator that starts from +0.
"""
import numpy as np
import pytest
import torch


def _state(rng, n, psi):
    master = np.zeros(n, np.float32)
    master[:psi] = rng.standard_normal(psi) * 0.02
    return master, np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)


def _micro(oracle_mod, rng, k, N, n, psi, sigma=1e-3, dtype="bf16"):
    out = []
    for _ in range(k):
        mb = []
        for _ in range(N):
            g = np.zeros(n, np.float32)
            g[:psi] = rng.standard_normal(psi) * sigma
            mb.append(oracle_mod.f32_to_bf16(g) if dtype == "bf16" else g)
        out.append(mb)
    return out


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("clip", [0.0, 0.01])
def test_one_micro_batch_is_the_plain_step(oracle_mod, dtype, clip):
    rng = np.random.default_rng(1)
    N, n, psi = 4, 4 * 128 * 3, 4 * 128 * 3 - 11
    hp = oracle_mod.Hparams(weight_decay=0.1, max_grad_norm=clip)
    a = _state(rng, n, psi)
    b = [x.copy() for x in a]
    for t in range(1, 4):
        mg = _micro(oracle_mod, rng, 1, N, n, psi, dtype=dtype)
        ra = oracle_mod.zero_step_accum(mg, *a, hp, t, 8.0)
        rb = oracle_mod.zero_step(mg[0], *b, hp, t, 8.0)
        assert ra == rb
        for x, y in zip(a, b):
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


@pytest.mark.parametrize("k,N", [(2, 4), (4, 2), (8, 8)])
def test_integer_micro_batches_equal_one_step_on_their_sums(oracle_mod, k, N):
    rng = np.random.default_rng(k * 10 + N)
    n = N * 128 * 2
    ints = rng.integers(-20, 21, size=(k, N, n))
    micro = [[oracle_mod.f32_to_bf16(ints[mb, r].astype(np.float32)) for r in range(N)]
             for mb in range(k)]
    summed = [ints[:, r].sum(axis=0).astype(np.float32) for r in range(N)]
    hp = oracle_mod.Hparams(lr=1e-3)
    a = _state(rng, n, n)
    b = [x.copy() for x in a]
    ra = oracle_mod.zero_step_accum(micro, *a, hp, 1, 2.0)
    rb = oracle_mod.zero_step(summed, *b, hp, 1, 2.0 * k)
    assert ra["applied"] and rb["applied"]
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


@pytest.mark.parametrize("k", [2, 5])
def test_n1_matches_torch_gradient_accumulation(oracle_mod, k):
    rng = np.random.default_rng(k)
    n = 128 * 64
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    master, m, v, w = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32), \
        np.zeros(n, np.uint16)
    tp = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    opt = torch.optim.AdamW([tp], lr=1e-3, weight_decay=0.1, foreach=False, fused=False)
    hp = oracle_mod.Hparams(lr=1e-3, weight_decay=0.1)
    for t in range(1, 6):
        micro = [[(rng.standard_normal(n) * 1e-3).astype(np.float32)] for _ in range(k)]
        oracle_mod.zero_step_accum(micro, master, m, v, w, hp, t, 1.0)
        tp.grad = None
        for mb in micro:
            g = torch.from_numpy(mb[0].copy()) / k
            tp.grad = g if tp.grad is None else tp.grad + g
        opt.step()
    def close(a, b, tol):
        rms = float(np.sqrt(np.mean(b.astype(np.float64) ** 2)))
        assert float(np.max(np.abs(a.astype(np.float64) - b))) <= tol * rms
    # m and v scale with the gradient (a dropped 1/k or a missing micro-batch
    # shows there); they must agree to FP32 rounding noise
    close(m, opt.state[tp]["exp_avg"].numpy(), 3e-6)
    close(v, opt.state[tp]["exp_avg_sq"].numpy(), 3e-6)
    # The weights: Adam's update g/(|g| + eps) is sensitive to the last bits of
    # accumulated gradients that nearly cancel (|g| ~ eps).  So they are
    # bounded in units of the update size, lr * steps.
    assert float(np.max(np.abs(master.astype(np.float64) - tp.detach().numpy()))) <= \
        1e-3 * hp.lr * 5


def test_nonfinite_in_any_micro_batch_skips(oracle_mod):
    rng = np.random.default_rng(4)
    N, n = 2, 2 * 128
    micro = _micro(oracle_mod, rng, 3, N, n, n)
    micro[1][1] = micro[1][1].copy()
    micro[1][1][17] = oracle_mod.f32_to_bf16(np.array([np.inf], np.float32))[0]
    st = _state(rng, n, n)
    before = [x.copy() for x in st]
    res = oracle_mod.zero_step_accum(micro, *st, oracle_mod.Hparams(), 1, 1.0, True)
    assert res["found_nonfinite"] and not res["applied"]
    for x, y in zip(st, before):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def test_micro_batches_add_in_order(oracle_mod):
    """N = 1, k = 4, loss scale 1, so each micro-batch adds its gradient times
    fp32(1/4) = 0.25 (exact).  Micro-batch values (T, 1, -T, 1) with T = 2**27
    add 2**25, 0.25, -2**25, 0.25.  In micro-batch order from +0:
    2**25, 2**25 + 0.25 = 2**25 (the FP32 spacing there is 4), +0, 0.25.
    Reversed: 0.25, -2**25 (spacing 2 just below), -2**25, +0.  In pairs:
    2**25 + -2**25 = +0.  m after one step from m = 0 is fp32(0.1) * g."""
    T = float(2 ** 27)
    n = 128
    micro = []
    for x in (T, 1.0, -T, 1.0):
        g = np.zeros(n, np.float32)
        g[0] = x
        micro.append([g])
    master, m, v, w = (np.zeros(n, np.float32), np.zeros(n, np.float32),
                       np.zeros(n, np.float32), np.zeros(n, np.uint16))
    res = oracle_mod.zero_step_accum(micro, master, m, v, w, oracle_mod.Hparams(), 1, 1.0)
    assert res["sumsq"] == 0.0625
    assert m[0] == np.float32(1.0 - 0.9) * np.float32(0.25)
    assert not m[1:].any()


def test_accumulator_starts_from_positive_zero(oracle_mod):
    """N = 1, k = 2, loss scale 1, FP32 gradients equal to -2**-149 (the
    negative subnormal of least magnitude) in both micro-batches.  Each
    contribution is -2**-149 * fp32(1/2) = -2**-150, a tie between -0 and
    -2**-149 that rounds to the even -0.  From +0 the accumulator is
    +0 + -0 = +0 twice over; started from the first contribution it would be
    -0.  With m = master = -0 before the step: m = 0.9 * -0 + 0.1 * +0 = +0 and
    master = -0 - lr * (+0 / eps) = -0 (a -0 gradient gives m = -0, master = +0)."""
    n = 2 * 128
    tiny = np.float32(-(2.0 ** -149))
    assert tiny != 0 and np.float32(tiny * np.float32(0.5)) == 0
    micro = [[np.full(n, tiny, np.float32)] for _ in range(2)]
    master = np.full(n, -0.0, np.float32)
    m = np.full(n, -0.0, np.float32)
    v = np.zeros(n, np.float32)
    w = np.zeros(n, np.uint16)
    res = oracle_mod.zero_step_accum(micro, master, m, v, w, oracle_mod.Hparams(), 1, 1.0)
    assert res["applied"] and res["sumsq"] == 0.0
    assert (m.view(np.uint32) == 0).all()
    assert (master.view(np.uint32) == 0x80000000).all()
    assert (w == 0x8000).all()
