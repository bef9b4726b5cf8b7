"""The oracle's all-cores timing mode (the same C source built with OpenMP)
against the single-thread build.

Every element is computed with the same operators in both builds, so the
state after a step is bit-identical whenever the norm does not enter it (no
clipping, or a clip coefficient of 1).  The step-wide sum of squares is added
in per-thread chunks in a fixed order, so it may differ from the sequential
sum in its last bits only; an active clip then stays within the parity
tolerance.
"""
import numpy as np
import pytest


@pytest.fixture(scope="module")
def omp(oracle_mod):
    try:
        oracle_mod.build(parallel=True)
    except Exception as exc:  # no OpenMP runtime for this compiler
        pytest.skip(f"the OpenMP build of the oracle is unavailable: {exc}")
    return oracle_mod


def _case(o, N, n, dtype, seed):
    rng = np.random.default_rng(seed)
    g = []
    for _ in range(N):
        x = (rng.standard_normal(n) * 32).astype(np.float32)
        g.append(o.f32_to_bf16(x) if dtype == "bf16" else x)
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    return g, p0


@pytest.mark.parametrize("N,dtype,clip,wd", [(8, "bf16", 0.0, 0.0), (4, "fp32", 0.0, 0.1),
                                             (3, "bf16", 1e9, 0.0), (4, "bf16", 1e-3, 0.0)])
def test_all_cores_build_matches_single_thread(omp, N, dtype, clip, wd):
    n = N * 128 * 3001
    g, p0 = _case(omp, N, n, dtype, N)
    hp = omp.Hparams(max_grad_norm=clip, weight_decay=wd)
    a = [p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)]
    b = [x.copy() for x in a]
    for t in (1, 2):
        ra = omp.zero_step(g, *a, hp, t, 1024.0, True)
        rb = omp.zero_step(g, *b, hp, t, 1024.0, True, parallel=True)
        assert ra["applied"] == rb["applied"] and ra["found_nonfinite"] == rb["found_nonfinite"]
        assert abs(ra["sumsq"] - rb["sumsq"]) <= 1e-12 * ra["sumsq"]
        if clip == 0.0 or ra["clip_coef"] == 1.0:
            for x, y in zip(a, b):
                assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
        else:
            assert abs(ra["clip_coef"] - rb["clip_coef"]) <= 1e-6 * ra["clip_coef"]
            np.testing.assert_allclose(b[0], a[0], rtol=1e-6, atol=1e-30)


def test_all_cores_build_flags_overflow(omp):
    N, n = 4, 4 * 128 * 1000
    g, p0 = _case(omp, N, n, "fp32", 7)
    g[2][n - 3] = np.inf
    st = [p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)]
    before = [x.copy() for x in st]
    res = omp.zero_step(g, *st, omp.Hparams(), 1, 1.0, True, parallel=True)
    assert res["found_nonfinite"] and not res["applied"]
    for x, y in zip(st, before):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
