"""Pins of the oracle's collective semantics and of the ZeRO step as a whole.

* reduce-scatter followed by all-gather equals all-reduce (the ledger page,
  "one full ZeRO-3 computation"; the DP-ZeRO blog, "three stages").
* The reduction adds the contributions of the same parameter only (RC-T2,
  note N48): poisoning other elements changes nothing.
* Brute force: integer-valued gradients make every sum exact, so the combined
  gradient is known by hand.
* The ZeRO step (owners update their slices, then all-gather) ends in exactly
  the state of the replicated DDP step on the same gradients (RC-T2, note
  N48: all ranks still train one model), bit for bit.
* Padding stays zero.
"""
import numpy as np
import pytest


def _grads(oracle_mod, rng, N, psi_pad, psi, dtype, sigma=1e-3):
    out = []
    for _ in range(N):
        g = np.zeros(psi_pad, np.float32)
        g[:psi] = rng.standard_normal(psi) * sigma
        out.append(oracle_mod.f32_to_bf16(g) if dtype == "bf16" else g)
    return out


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("units", [1, 3])
def test_reduce_scatter_then_all_gather_is_all_reduce(oracle_mod, N, dtype, units):
    rng = np.random.default_rng(N * 10 + units)
    psi_pad = units * N * 128
    grads = _grads(oracle_mod, rng, N, psi_pad, psi_pad - 5, dtype)
    inv = np.float32(1.0 / N)
    shards = [oracle_mod.reduce_scatter(grads, psi_pad, r, inv) for r in range(N)]
    assert all(s.size == psi_pad // N for s in shards)
    gathered = oracle_mod.all_gather_f32(shards)
    full = oracle_mod.all_reduce(grads, psi_pad, inv)
    assert np.array_equal(gathered.view(np.uint32), full.view(np.uint32))


@pytest.mark.parametrize("N", [2, 4, 7])
def test_integer_gradients_brute_force(oracle_mod, N):
    """Small integers are exact in BF16 and their sums are exact in FP32; with
    N a power of two (or any N, by checking N * g) the mean is known exactly."""
    rng = np.random.default_rng(N)
    psi_pad = 2 * N * 128
    ints = rng.integers(-100, 101, size=(N, psi_pad))
    grads = [oracle_mod.f32_to_bf16(row.astype(np.float32)) for row in ints]
    for loss_scale in (1.0, 4.0):
        inv = np.float32(1.0 / (N * loss_scale))
        full = oracle_mod.all_reduce(grads, psi_pad, inv)
        total = ints.sum(axis=0)
        expected = (total.astype(np.float32) * inv)  # one rounding of an exact integer sum
        assert np.array_equal(full, expected)
        if N & (N - 1) == 0:
            assert np.array_equal(full.astype(np.float64), total / (N * loss_scale))


@pytest.mark.parametrize("N", [2, 4])
def test_same_parameter_only(oracle_mod, N):
    rng = np.random.default_rng(11)
    psi_pad = 2 * N * 128
    shard = psi_pad // N
    grads = _grads(oracle_mod, rng, N, psi_pad, psi_pad, "fp32")
    inv = np.float32(1.0 / N)
    for r in range(N):
        ref = oracle_mod.reduce_scatter(grads, psi_pad, r, inv)
        poisoned = [g.copy() for g in grads]
        for g in poisoned:
            g[: r * shard] = np.nan
            g[(r + 1) * shard:] = np.inf
        assert np.array_equal(oracle_mod.reduce_scatter(poisoned, psi_pad, r, inv), ref)
        # changing one element of the slice changes that element only
        poisoned[N - 1][r * shard + 3] += np.float32(1.0)
        got = oracle_mod.reduce_scatter(poisoned, psi_pad, r, inv)
        diff = np.flatnonzero(got != ref)
        assert diff.tolist() == [3]


def _fresh_state(rng, psi_pad, psi):
    master = np.zeros(psi_pad, np.float32)
    master[:psi] = rng.standard_normal(psi) * 0.02
    return master, np.zeros(psi_pad, np.float32), np.zeros(psi_pad, np.float32), \
        np.zeros(psi_pad, np.uint16)


CASES = [
    dict(N=4, dtype="bf16", wd=0.0, clip=0.0, scale=1.0),
    dict(N=3, dtype="fp32", wd=0.1, clip=0.0, scale=1.0),
    dict(N=8, dtype="bf16", wd=0.0, clip=0.0, scale=65536.0),
    dict(N=4, dtype="fp32", wd=0.0, clip=0.05, scale=1.0),
    dict(N=2, dtype="bf16", wd=0.1, clip=1.0, scale=8.0),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_zero_step_equals_ddp_step(oracle_mod, case):
    N = case["N"]
    rng = np.random.default_rng(N + 100)
    psi = 2 * N * 128 + 37
    psi_pad = 3 * N * 128
    hp = oracle_mod.Hparams(lr=1e-3, weight_decay=case["wd"], max_grad_norm=case["clip"])
    master, m, v, w = _fresh_state(rng, psi_pad, psi)
    reps = [[a.copy() for _ in range(N)] for a in (master, m, v, w)]
    for t in range(1, 5):
        grads = _grads(oracle_mod, rng, N, psi_pad, psi, case["dtype"],
                       sigma=1e-3 * case["scale"])
        rz = oracle_mod.zero_step(grads, master, m, v, w, hp, t, case["scale"])
        rd = oracle_mod.ddp_step(grads, *reps, hp, t, case["scale"])
        assert rz == rd
        for full, rep in zip((master, m, v, w), reps):
            for i in range(N):
                assert np.array_equal(full.view(np.uint8), rep[i].view(np.uint8))
    # padding stays exactly zero in every state array and in the weights
    for a in (master, m, v, w):
        assert not a[psi:].view(np.uint8).any()
    # the working weights are the all-gathered BF16 rounding of the master
    assert np.array_equal(w, oracle_mod.f32_to_bf16(master))
