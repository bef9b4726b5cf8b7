"""GPU parity on gradients crafted so that the result depends on the order of
the reduction and on its start value.

The combined gradient is the FP32 sum of the N contributions in rank order
0..N-1, from +0, then one multiply by fp32(1/(N * loss_scale)); an
accumulated step adds its micro-batches' parts in order to an accumulator
that starts from +0.  The oracle's pins (tests/test_oracle_collectives.py,
tests/test_oracle_accum.py) fix that order by hand-worked FP32 cases.  Here
every kernel form of the CUDA path runs on the same crafted columns and must
match the oracle bit for bit.  With T = 2**27:
  pattern 0, ranks (1, T, -T, +0 ...): +0 in rank order (1 in reverse);
  pattern 1, ranks (T, 1, -T, 1, +0 ...): 1 in rank order (+0 in reverse or
             in pairs);
  pattern 2, every rank -0, with master = m = -0: the sum from +0 is +0, so
             m becomes +0 and master stays -0 (w = 0x8000);
  pattern 3, ordinary N(0, sigma) gradients;
  pattern 4, rank 0 the negative subnormal of least magnitude, the others +0:
             the scaled combined gradient rounds to -0, so m = 0.9 * -0 +
             0.1 * -0 stays -0 in a one-batch step; an accumulator that starts
             from +0 turns it into +0.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from parity_util import compare_result, compare_state, state_to_numpy

pytestmark = pytest.mark.gpu

T27 = float(2 ** 27)
LOSS_SCALE = 65536.0


def _crafted_grads(N, psi_pad, dtype, seed, sigma=1e-3 * LOSS_SCALE):
    """N rank buffers (torch, CPU) with the five patterns by element index mod 5."""
    j = np.arange(psi_pad)
    pat = j % 5
    rng = np.random.default_rng(seed)
    # least-magnitude negative subnormal of the gradient type
    tiny = -(2.0 ** -133) if dtype == "bf16" else -(2.0 ** -149)
    rows = np.zeros((N, psi_pad), np.float32)
    col0 = [1.0, T27, -T27]
    col1 = [T27, 1.0, -T27, 1.0]
    for i in range(N):
        if i < len(col0):
            rows[i, pat == 0] = col0[i]
        if N >= 4 and i < len(col1):
            rows[i, pat == 1] = col1[i]
        rows[i, pat == 2] = -0.0
        rows[i, pat == 3] = rng.standard_normal(int((pat == 3).sum())) * sigma
        if i == 0:
            rows[i, pat == 4] = tiny
    if N < 3:   # too few ranks for the order patterns: ordinary values there
        for i in range(N):
            rows[i, pat <= 1] = rng.standard_normal(int((pat <= 1).sum())) * sigma
    t = torch.from_numpy(rows)
    out = [t[i].clone() for i in range(N)]
    if dtype == "bf16":
        out = [x.to(torch.bfloat16) for x in out]
    assert float(out[0][4].float()) == tiny   # the subnormal survives the cast
    return out, pat


def _np(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _initial_state(psi_pad, pat, seed):
    g = torch.Generator().manual_seed(seed)
    master = torch.randn(psi_pad, generator=g) * 0.02
    m = torch.randn(psi_pad, generator=g).abs() * 1e-4
    v = torch.rand(psi_pad, generator=g) * 1e-8
    zero_sign = torch.from_numpy(pat == 2) | torch.from_numpy(pat == 4)
    master[zero_sign] = -0.0
    m[zero_sign] = -0.0
    v[zero_sign] = 0.0
    w = torch.zeros(psi_pad, dtype=torch.int16)
    return master, m, v, w


FORMS = {
    "fused-in-place": dict(),
    "fused-out-of-place-skip": dict(out_of_place=True, skip=True),
    "staged-in-place": dict(staging=1),
    "staged-out-of-place-policy": dict(out_of_place=True, skip=True, staging=1, policy=True),
    "staged-pingpong-policy": dict(out_of_place=True, skip=True, staging=1, policy=True,
                                   pingpong=True),
    "two-pass-in-place-skip": dict(skip=True),
    "two-pass-clip": dict(clip=1e9, out_of_place=True),
    "buckets": dict(bucket=4096, skip=True, out_of_place=True),
    "accumulate-fused-last": dict(micro=2, out_of_place=True),
    "accumulate-two-pass": dict(micro=3, skip=True),
}


@pytest.mark.parametrize("form", list(FORMS))
@pytest.mark.parametrize("N,dtype", [(1, "bf16"), (2, "fp32"), (3, "bf16"), (4, "bf16"),
                                     (4, "fp32"), (5, "fp32"), (8, "bf16")])
def test_crafted_columns_match_the_oracle(zero_lib, oracle_mod, form, N, dtype):
    from zero_sharded_mixed_04_gb300.optim import ZeroAdam
    f = FORMS[form]
    dev = torch.device("cuda:0")
    psi_pad = N * 128 * 41          # several 2048-element tiles and a ragged last tile
    k = f.get("micro", 0)
    clip = f.get("clip", 0.0)
    opt = ZeroAdam(psi_pad, N, dtype, skip_on_overflow=f.get("skip", False), max_grad_norm=clip,
                   bucket_elems=f.get("bucket", 0), loss_scale=LOSS_SCALE,
                   out_of_place=f.get("out_of_place", False), device=dev,
                   smem_staging=f.get("staging", 0), micro_batches=k,
                   device_policy=f.get("policy", False), pingpong=f.get("pingpong", False))
    grads, pat = _crafted_grads(N, psi_pad, dtype, seed=N)
    master, m, v, w = _initial_state(psi_pad, pat, seed=10 + N)
    opt.load_state(master.to(dev), m.to(dev), v.to(dev), w.to(dev))
    ref = {"master": master.numpy().copy(), "m": m.numpy().copy(), "v": v.numpy().copy(),
           "w": w.numpy().view(np.uint16).copy()}
    hp = oracle_mod.Hparams(max_grad_norm=clip)
    for step in (1, 2):
        if k:
            micro = [grads] + [_crafted_grads(N, psi_pad, dtype, seed=100 * step + mb)[0]
                               for mb in range(1, k)]
            res = opt.step_accumulated([[g.to(dev) for g in mb] for mb in micro])
            ores = oracle_mod.zero_step_accum([[_np(g) for g in mb] for mb in micro],
                                              ref["master"], ref["m"], ref["v"], ref["w"], hp,
                                              step, LOSS_SCALE, f.get("skip", False))
        else:
            res = opt.step([g.to(dev) for g in grads])
            ores = oracle_mod.zero_step([_np(g) for g in grads], ref["master"], ref["m"],
                                        ref["v"], ref["w"], hp, step, LOSS_SCALE,
                                        f.get("skip", False))
        compare_result(res, ores)
        assert ores["applied"] and res["applied"]
        got = state_to_numpy(opt.state())
        # clip at 1e9 never clips (coef = 1), so every form is bit-exact
        compare_state(got, ref, exact=True, tag=f"{form} step {step} ")
        if step == 1:
            # the hand-worked facts, independently of the oracle
            m_bits = got["m"].view(np.uint32)
            p_bits = got["master"].view(np.uint32)
            assert (m_bits[pat == 2] == 0).all(), "a sum of -0 contributions from +0 is +0"
            assert (p_bits[pat == 2] == 0x80000000).all()
            assert (got["w"][pat == 2] == 0x8000).all()
            if N >= 2:
                # one batch: the scaled gradient is -0 and m stays -0; an
                # accumulator from +0 gives +0
                want = 0 if k else 0x80000000
                assert (m_bits[pat == 4] == want).all()
