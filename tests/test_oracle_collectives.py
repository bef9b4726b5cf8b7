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
* The reduction order and its start: hand-worked FP32 cases whose bits
  depend on the ranks being added in order 0..N-1 from +0.
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


# ---------------------------------------------------------------------------
# Reduction order and start value.
#
# The combined gradient is the FP32 sum of the ranks' contributions taken in
# rank order 0..N-1, starting from +0 (RC-T2 note N48: the reduction adds the
# contributions of one parameter; the order and the start are this library's
# reading, since the pages do not fix them).  The cases below make every other
# order or start give different bits.  Every expected value is worked out by
# hand from IEEE round-to-nearest-even FP32 addition:
#   T = 2**27 is exact in BF16 and FP32.  Next to it the FP32 spacing is 16
#   above and 8 below, so T + 1 rounds back to T and -T + 1 back to -T.  An
#   exact zero sum of non-zero terms is +0, and +0 + -0 = +0, -0 + -0 = -0.
# ---------------------------------------------------------------------------

T27 = float(2 ** 27)


def _crafted(oracle_mod, rows, dtype, N, psi_pad):
    """Rank buffers whose first len(rows[0]) elements are the given columns
    (rows[i] is rank i's values), the rest +0."""
    out = []
    for i in range(N):
        g = np.zeros(psi_pad, np.float32)
        g[:len(rows[i])] = rows[i]
        out.append(oracle_mod.f32_to_bf16(g) if dtype == "bf16" else g)
    return out


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_reduction_is_in_rank_order(oracle_mod, dtype):
    # Four columns, N = 4 ranks, listed as (rank 0, rank 1, rank 2, rank 3):
    # column 0 (1, T, -T, +0): 1, 1 + T = T, T - T = +0, +0 -> +0.
    #   Reversed: +0, -T, +0, 1 -> 1.
    # column 1 (T, 1, -T, +0): T, T, +0, +0 -> +0 (reversed too).
    # column 2 (T, 1, -T, 1): T, T + 1 = T, +0, +0 + 1 = 1.
    #   In pairs: (T + 1) + (-T + 1) = T + -T = +0.  Reversed: 1, 1 - T = -T,
    #   -T + 1 = -T, -T + T = +0.  Only the rank order gives 1.
    # column 3 (1, -T, T, 1): 1, -T, +0, 1 -> 1, in every order (a control).
    N = 4
    psi_pad = N * 128
    rows = [[1.0, T27, T27, 1.0],
            [T27, 1.0, 1.0, -T27],
            [-T27, -T27, -T27, T27],
            [0.0, 0.0, 1.0, 1.0]]
    grads = _crafted(oracle_mod, rows, dtype, N, psi_pad)
    got = oracle_mod.all_reduce(grads, psi_pad, np.float32(1.0))
    want = np.array([0.0, 0.0, 1.0, 1.0], np.float32)
    assert np.array_equal(got[:4].view(np.uint32), want.view(np.uint32)), got[:4]
    assert not got[4:].view(np.uint32).any()
    # the batch mean: one multiply by fp32(1/4) = 0.25 (exact)
    got = oracle_mod.all_reduce(grads, psi_pad, np.float32(0.25))
    assert got[:4].tolist() == [0.0, 0.0, 0.25, 0.25]
    # three ranks: column 0 of the first three ranks, (1, T, -T) -> +0
    g3 = _crafted(oracle_mod, [r[:1] for r in rows[:3]], dtype, 3, 3 * 128)
    got = oracle_mod.all_reduce(g3, 3 * 128, np.float32(1.0 / 3.0))
    assert got[0] == 0.0 and got.view(np.uint32)[0] == 0
    # every owner's slice sums in the same order: the same column placed at the
    # start of each owner's slice gives the same bits
    shard = psi_pad // N
    for r in range(N):
        g = []
        for i in range(N):
            x = np.zeros(psi_pad, np.float32)
            x[r * shard + 7] = rows[i][2]
            g.append(oracle_mod.f32_to_bf16(x) if dtype == "bf16" else x)
        sl = oracle_mod.reduce_scatter(g, psi_pad, r, np.float32(1.0))
        assert sl[7] == 1.0 and np.count_nonzero(sl) == 1


@pytest.mark.parametrize("N", [1, 2, 3, 8])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_reduction_starts_from_positive_zero(oracle_mod, N, dtype):
    """Every rank contributing -0: a sum started from +0 is +0 (+0 + -0 = +0),
    while a sum started from rank 0's value would stay -0."""
    psi_pad = N * 128
    grads = []
    for _ in range(N):
        g = np.full(psi_pad, -0.0, np.float32)
        grads.append(oracle_mod.f32_to_bf16(g) if dtype == "bf16" else g)
    if dtype == "bf16":
        assert (grads[0] == 0x8000).all()
    full = oracle_mod.all_reduce(grads, psi_pad, np.float32(1.0 / N))
    assert (full.view(np.uint32) == 0).all()


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_step_sees_the_sign_of_a_zero_sum(oracle_mod, dtype):
    """One step with every gradient -0 and master = m = -0, v = +0, t = 1, no
    weight decay.  The combined gradient is +0 (the sum starts from +0), so
      m = 0.9 * -0 + 0.1 * +0 = -0 + +0 = +0,
      den = sqrt(+0) / sqrt(1 - 0.999) + eps = eps,  m / den = +0,
      master = -0 - lr * (+0) = -0 + -0 = -0,  w = bf16(-0) = 0x8000.
    A combined gradient of -0 would give m = -0 and master = -0 - (-0) = +0."""
    N = 4
    psi_pad = N * 128
    grads = []
    for _ in range(N):
        g = np.full(psi_pad, -0.0, np.float32)
        grads.append(oracle_mod.f32_to_bf16(g) if dtype == "bf16" else g)
    master = np.full(psi_pad, -0.0, np.float32)
    m = np.full(psi_pad, -0.0, np.float32)
    v = np.zeros(psi_pad, np.float32)
    w = np.zeros(psi_pad, np.uint16)
    res = oracle_mod.zero_step(grads, master, m, v, w, oracle_mod.Hparams(), 1, 1.0, True)
    assert res["applied"] and not res["found_nonfinite"] and res["sumsq"] == 0.0
    assert (m.view(np.uint32) == 0x00000000).all()
    assert (v.view(np.uint32) == 0x00000000).all()
    assert (master.view(np.uint32) == 0x80000000).all()
    assert (w == 0x8000).all()


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_step_uses_the_rank_order_sum(oracle_mod, dtype):
    """The same crafted columns through the whole step: m after one step from
    m = 0 is fp32(0.1) * g, so it shows g itself.  Column 0 (1, T, -T, +0)
    must leave m at +0 and column 2 (T, 1, -T, 1) at fp32(0.1) * 0.25."""
    N = 4
    psi_pad = N * 128
    rows = [[1.0, T27], [T27, 1.0], [-T27, -T27], [0.0, 1.0]]
    grads = _crafted(oracle_mod, rows, dtype, N, psi_pad)
    master = np.zeros(psi_pad, np.float32)
    m = np.zeros(psi_pad, np.float32)
    v = np.zeros(psi_pad, np.float32)
    w = np.zeros(psi_pad, np.uint16)
    oracle_mod.zero_step(grads, master, m, v, w, oracle_mod.Hparams(), 1, 1.0)
    omb1 = np.float32(1.0 - 0.9)
    assert m.view(np.uint32)[0] == 0
    assert m[1] == omb1 * np.float32(0.25)
    # first step from m = v = 0: the update is -lr * g / (|g| + eps) (exactly
    # -lr * 1 / (1 + eps/|g|)), so master moves by about -lr where g > 0 and
    # not at all where g = 0
    assert master[0] == 0.0
    assert abs(master[1] + 1e-3) < 1e-8
