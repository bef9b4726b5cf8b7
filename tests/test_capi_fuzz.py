"""The C ABI's argument checks under seeded random arguments, on the host.

Every entry point is called with sizes, counts, dtypes, hyper-parameters,
alignments, overlaps and workspace sizes drawn at random, many of them
invalid: huge and negative sizes, counts past ZERO_MAX_ELEMS, misaligned and
overlapping buffers, too-small workspaces.  The addresses are made up, so no
call may reach a kernel with them; on this host, with no GPU, a call whose
arguments all pass reaches the CUDA runtime and gets ZERO_ERR_CUDA back.  The
process must survive every call, and each must return one of the codes the
header documents for it.  Each case runs in a child process, so a crash fails
its case instead of the run.

Only run without a GPU: with one, arguments that pass the checks would launch
kernels on made-up addresses.
"""
from __future__ import annotations

import json
import os
import random
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GB = 1 << 30
SEEDS = 400


def _no_gpu() -> bool:
    import torch
    return not torch.cuda.is_available()


pytestmark = pytest.mark.skipif(not _no_gpu(), reason="made-up addresses: host-only test")

CHILD = r'''
import ctypes, json, random, sys
sys.path.insert(0, ROOT)
from zero_sharded_mixed_04_gb300 import zero as Z
GB = 1 << 30
MAXE = Z.ZERO_MAX_ELEMS

def addr(r, base):
    a = base
    if r.random() < 0.1:
        a += r.choice([1, 2, 4, 8])          # misaligned
    return None if r.random() < 0.03 else a

def size(r, unit):
    return r.choice([0, -unit, unit, 3 * unit, 1 << 20, r.randrange(1, 1 << 22) * unit,
                     MAXE, MAXE + unit, 1 << 62, (1 << 63) - 1, -(1 << 63), unit + 8])

def case(seed):
    r = random.Random(seed)
    out = []
    for _ in range(25):
        N = r.choice([-1, 0, 1, 2, 3, 4, 8, 16, 64, 65, 1000])
        n_ok = max(1, min(N, 64))
        psi_pad = size(r, max(1, N) * 128)
        dtype = r.choice([0, 1, 1, 2, -1])
        hp = Z.make_hparams(lr=r.choice([1e-3, -1.0, float("nan")]),
                            beta1=r.choice([0.9, 1.0]), beta2=r.choice([0.999, -0.1]),
                            eps=r.choice([1e-8, 0.0]), weight_decay=r.choice([0.0, 0.1]),
                            max_grad_norm=r.choice([0.0, 1.0, -1.0]),
                            step=r.choice([1, 0, 5]), skip_on_overflow=r.random() < 0.5,
                            bucket_elems=r.choice([0, 8, 12, 1 << 20, -8]),
                            micro_batches=r.choice([0, 1, 2, -1]))
        base = [addr(r, (6 + i) * GB) for i in range(n_ok)]
        if r.random() < 0.1 and n_ok > 1:
            base[1] = base[0]                  # two ranks share a buffer
        st = [addr(r, k * GB) for k in (1, 2, 3, 4)]
        dst = [addr(r, k * GB) for k in (10, 11, 12, 13)] if r.random() < 0.5 else st
        if r.random() < 0.1:
            dst = [st[0]] + dst[1:]            # src and dst share master
        ws = addr(r, 5 * GB) if r.random() < 0.95 else 5 * GB + 16
        need = Z.zero_workspace_bytes(psi_pad, hp, dst is st)
        ws_bytes = r.choice([need, max(0, need - 1), 0, need + (1 << 20), 16640])
        ls = r.choice([1.0, 0.0, -1.0, float("inf"), float("nan"), 65536.0])
        which = r.choice(["step", "into", "plan", "noalloc", "ws", "layout", "ledger",
                          "gather", "peak", "comm", "table"])
        if which == "step":
            rc = Z.zero_step(base, dtype, *st, psi_pad, N, hp, ls, ws, ws_bytes, None, 0)
        elif which == "into":
            rc = Z.zero_step_into(base, dtype, *st, *dst, psi_pad, N, hp, ls, ws, ws_bytes,
                                  None, 0)
        elif which == "noalloc":
            rc = Z.zero_step_noalloc(base, dtype, *st, psi_pad, N, hp, ls, None, 0)
        elif which == "plan":
            plan = Z.zero_plan()
            rc = Z.zero_plan_init(plan, base, dtype, *st, *dst, psi_pad, N, hp, ls, ws, ws_bytes)
            if rc == Z.ZERO_OK:
                # no device: begin fails in the runtime; buckets and end before
                # a begin are refused on the host
                rc2 = Z.zero_plan_bucket(plan, 0, max(8, psi_pad), None, 0)
                rc3 = Z.zero_plan_end(plan, None, 0)
                # made-up policy and table addresses: no device maps them
                rc4 = Z.zero_plan_set_device_policy_table(plan, 9 * GB, 9 * GB + 4096,
                                                          r.choice([1, 0, MAXE]),
                                                          r.choice([1, 64, 0, -1]))
                out.append(["plan_policy_table", rc4])
                rc = Z.zero_plan_begin(plan, 0)
                out.append(["plan_bucket_before_begin", rc2])
                out.append(["plan_end_before_begin", rc3])
        elif which == "ws":
            rc = Z.zero_workspace_bytes(psi_pad, hp, r.random() < 0.5)
            rc = "zero" if rc == 0 else ("ok" if rc > 0 else "negative")
        elif which == "layout":
            sizes = [r.choice([0, 1, 7, 1 << 20, -1, MAXE, 1 << 62]) for _ in range(r.randrange(0, 6))]
            rc, lay, offs = Z.zero_init_layout(sizes, N)
            if rc == Z.ZERO_OK:
                assert lay.psi_pad <= MAXE and lay.psi_pad % (N * 128) == 0, (sizes, N)
                assert lay.psi == sum(sizes)
        elif which == "ledger":
            v = Z._lib.zero_ledger(size(r, 1), N, r.choice([-1, 0, 1, 2, 3, 4]),
                                   r.choice([-1, 2, 4, 100]), r.choice([12, 8, 1000]))
            rc = "neg1" if v == -1 else ("ok" if v >= 0 else "negative")
        elif which == "comm":
            v = Z._lib.zero_comm_volume(size(r, 1), N, r.choice([-1, 0, 1, 2, 3, 4]))
            rc = "neg1" if v == -1 else ("ok" if v >= 0 else "negative")
        elif which == "peak":
            layers = [r.choice([0, 1, 1 << 20, -1, MAXE, 1 << 62]) for _ in range(r.randrange(0, 5))]
            v = Z.zero3_peak_bytes(layers, N)
            rc = "neg1" if v == -1 else ("ok" if v >= 0 else "negative")
        elif which == "table":
            # the table is written: a real buffer for the counts the library
            # may accept, a made-up address only for counts it must refuse
            t_first = r.choice([-1, 0, 1, 5, MAXE, MAXE + 1, 1 << 62])
            t_count = r.choice([-1, 0, 1, 7, MAXE + 1, 1 << 62, -(1 << 63)])
            if 1 <= t_count <= 7:
                buf = (ctypes.c_float * (2 * t_count))()
                rc = Z.zero_policy_table_fill(hp, t_first, t_count, ctypes.addressof(buf))
            else:
                rc = Z.zero_policy_table_fill(hp, t_first, t_count, 7 * GB)
        else:
            shard = size(r, 8)
            rc = Z.zero3_gather(base, N, shard, r.choice([0, 5, -1, 8]),
                                r.choice([0, 8, 1 << 20, shard, 1 << 62]), ws, 0, 0)
        out.append([which, rc])
    return out

print(json.dumps(case(int(sys.argv[1]))))
'''

ALLOWED = {
    "step": {0, -1, -2, -3, -5, -6, 1}, "into": {0, -1, -2, -3, -5, -6, 1},
    "noalloc": {0, -1, -2, -3, -5, -6, -7, 1}, "plan": {0, -1, -2, -3, -5, -6},
    "plan_bucket_before_begin": {-1}, "plan_end_before_begin": {-1}, "plan_policy_table": {-1},
    "table": {0, -1},
    "ws": {"zero", "ok"}, "layout": {0, -1}, "ledger": {"neg1", "ok"},
    "comm": {"neg1", "ok"}, "peak": {"neg1", "ok"}, "gather": {0, -1, -2, -3, -6},
}


@pytest.mark.parametrize("block", range(8))
def test_random_arguments_never_crash(block, tmp_path):
    """Each block runs SEEDS / 8 child processes of 25 calls each."""
    script = tmp_path / "child.py"
    script.write_text(CHILD.replace("ROOT", repr(ROOT)))
    for seed in range(block, SEEDS, 8):
        r = subprocess.run([sys.executable, str(script), str(seed)], capture_output=True,
                           text=True, timeout=120, env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
        assert r.returncode == 0, f"seed {seed}: the process died\n{r.stderr[-2000:]}"
        for which, rc in json.loads(r.stdout.strip().splitlines()[-1]):
            assert rc in ALLOWED[which], f"seed {seed}: {which} returned {rc!r}"


def test_sizes_past_the_limit_are_refused():
    from zero_sharded_mixed_04_gb300 import zero as Z
    big = Z.ZERO_MAX_ELEMS + 4 * 128
    hp = Z.make_hparams()
    assert Z.zero_workspace_bytes(big, hp, True) == 0
    assert Z.zero_workspace_bytes(Z.ZERO_MAX_ELEMS, hp, True) > 0
    grads = [6 * GB + i * GB for i in range(4)]
    assert Z.zero_step(grads, Z.ZERO_GRAD_BF16, 1 * GB, 2 * GB, 3 * GB, 4 * GB, big, 4, hp, 1.0,
                       5 * GB, 1 << 40, None, 0) == Z.ZERO_ERR_ARG
    assert Z.zero_init_layout([Z.ZERO_MAX_ELEMS, 1], 4)[0] == Z.ZERO_ERR_ARG
    assert Z.zero_init_layout([1 << 62, 1 << 62], 4)[0] == Z.ZERO_ERR_ARG
    assert Z._lib.zero_ledger(Z.ZERO_MAX_ELEMS + 1, 4, 0, 2, 12) == -1
    assert Z._lib.zero_ledger(Z.ZERO_MAX_ELEMS, 4, 0, 2, 12) == 16 * Z.ZERO_MAX_ELEMS
    assert Z._lib.zero_comm_volume((1 << 62), 4, 3) == -1
    assert Z.zero3_peak_bytes([1 << 62, 1 << 62], 4) == -1
    assert Z.zero3_gather(grads, 4, Z.ZERO_MAX_ELEMS, 0, 8, 5 * GB, 0, 0) == Z.ZERO_ERR_ARG
