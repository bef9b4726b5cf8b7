"""The C-ABI library on the host: it loads, exports every function the header
declares, and its host-only entry points (layout, ledger, communication
count, argument checking) agree with the oracle.  No GPU work is launched:
every zero_step call here fails argument validation before enqueueing."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(zero3?_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("zero_init_layout", "zero_step", "zero_ledger", "zero_workspace_bytes"):
        assert required in names


def test_library_exports_every_declared_symbol(zero_lib):
    lib = ctypes.CDLL(zero_lib.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    assert sorted(zero_lib.exported_symbols()) == _declared_functions()


@pytest.mark.parametrize("numel,N", [([1], 1), ([3, 5, 7], 4), ([128] * 8, 8), ([1000, 24], 3),
                                     ([], 2), ([50257 * 768, 768, 768], 4), ([5], 64)])
def test_layout_matches_oracle(zero_lib, oracle_mod, numel, N):
    rc, lay, offs = zero_lib.zero_init_layout(numel, N)
    assert rc == zero_lib.ZERO_OK
    o_offs, psi, psi_pad, shard = oracle_mod.layout(numel, N)
    assert (lay.psi, lay.psi_pad, lay.shard, lay.N, lay.n_tensors) == (psi, psi_pad, shard, N,
                                                                        len(numel))
    assert list(offs) == list(o_offs)
    for r in range(N):
        rc, b, e = zero_lib.zero_shard_range(lay, r)
        assert rc == 0 and (b, e) == (r * shard, (r + 1) * shard)
    assert zero_lib.zero_shard_range(lay, N)[0] == zero_lib.ZERO_ERR_ARG


def test_layout_rejects_bad_arguments(zero_lib):
    assert zero_lib.zero_init_layout([1, -1], 2)[0] == zero_lib.ZERO_ERR_ARG
    assert zero_lib.zero_init_layout([1], 0)[0] == zero_lib.ZERO_ERR_ARG
    assert zero_lib.zero_init_layout([1], 65)[0] == zero_lib.ZERO_ERR_ARG


@pytest.mark.parametrize("psi", [0, 1, 10, 8_000_000_000, 7_000_000_000, 123_588_864])
@pytest.mark.parametrize("N", [1, 3, 4, 8])
@pytest.mark.parametrize("stage", [0, 1, 2, 3])
@pytest.mark.parametrize("gb,ob", [(2, 12), (4, 12), (2, 8)])
def test_ledger_and_comm_match_oracle(zero_lib, oracle_mod, psi, N, stage, gb, ob):
    assert zero_lib.zero_ledger(psi, N, stage, gb, ob) == oracle_mod.ledger_bytes(psi, N, stage,
                                                                                   gb, ob)
    assert zero_lib.zero_comm_volume(psi, N, stage) == oracle_mod.comm_volume(psi, N, stage)


def test_ledger_printed_values(zero_lib):
    assert [zero_lib.zero_ledger(8_000_000_000, 4, s) for s in range(4)] == \
        [128_000_000_000, 56_000_000_000, 44_000_000_000, 32_000_000_000]
    assert zero_lib.zero_ledger(-1, 4, 0) == -1 and zero_lib.zero_ledger(1, 4, 4) == -1


def test_workspace_bytes(zero_lib):
    Z = zero_lib
    hp = Z.make_hparams()
    base = Z.zero_workspace_bytes(1 << 20, hp, True)
    assert base > 0 and base % 256 == 0
    hp_skip = Z.make_hparams(skip_on_overflow=True)
    # in place with skip needs the FP32 combined gradient; out of place does not
    assert Z.zero_workspace_bytes(1 << 20, hp_skip, True) == base + 4 * (1 << 20)
    assert Z.zero_workspace_bytes(1 << 20, hp_skip, False) == base
    hp_clip = Z.make_hparams(max_grad_norm=1.0)
    assert Z.zero_workspace_bytes(1 << 20, hp_clip, False) == base + 4 * (1 << 20)
    assert Z.zero_workspace_bytes(-1, hp, True) == 0


def test_status_strings(zero_lib):
    Z = zero_lib
    for code in (Z.ZERO_OK, Z.ZERO_STEP_SKIPPED, Z.ZERO_ERR_ARG, Z.ZERO_ERR_ALIGN, Z.ZERO_ERR_CUDA,
                 Z.ZERO_ERR_TIMEOUT, Z.ZERO_ERR_WORKSPACE, Z.ZERO_ERR_OVERLAP):
        assert Z.zero_status_str(code) != "unknown status"
    assert Z.zero_status_str(12345) == "unknown status"


# ---------------------------------------------------------------- argument checking
# Fake device addresses: every call below must be rejected before any CUDA call.

GB = 1 << 30


def _call(Z, N=4, psi_pad=4 * 128 * 4, grads=None, master=1 * GB, m=2 * GB, v=3 * GB, w=4 * GB,
          ws=5 * GB, ws_bytes=None, hp=None, loss_scale=1.0, dtype=None):
    hp = hp or Z.make_hparams()
    grads = grads if grads is not None else [6 * GB + i * GB // 4 for i in range(N)]
    ws_bytes = Z.zero_workspace_bytes(psi_pad, hp, True) if ws_bytes is None else ws_bytes
    return Z.zero_step(grads, Z.ZERO_GRAD_BF16 if dtype is None else dtype, master, m, v, w,
                       psi_pad, N, hp, loss_scale, ws, ws_bytes, None, 0)


def test_step_rejects_bad_sizes(zero_lib):
    Z = zero_lib
    assert _call(Z, N=0, grads=[]) == Z.ZERO_ERR_ARG
    assert _call(Z, N=65, grads=[6 * GB] * 65) == Z.ZERO_ERR_ARG
    assert _call(Z, psi_pad=4 * 128 * 4 + 8) == Z.ZERO_ERR_ARG      # not a multiple of N*128
    assert _call(Z, psi_pad=-512) == Z.ZERO_ERR_ARG
    assert _call(Z, dtype=7) == Z.ZERO_ERR_ARG
    assert _call(Z, loss_scale=0.0) == Z.ZERO_ERR_ARG
    assert _call(Z, loss_scale=float("inf")) == Z.ZERO_ERR_ARG


@pytest.mark.parametrize("field,value", [("lr", -1.0), ("beta1", 1.0), ("beta2", -0.1),
                                         ("eps", 0.0), ("weight_decay", float("nan")),
                                         ("max_grad_norm", -1.0), ("step", 0),
                                         ("skip_on_overflow", 2), ("micro_batches", -1),
                                         ("bucket_elems", 12)])
def test_step_rejects_bad_hparams(zero_lib, field, value):
    Z = zero_lib
    hp = Z.make_hparams()
    setattr(hp, field, value)
    assert _call(Z, hp=hp, ws_bytes=1 << 30) == Z.ZERO_ERR_ARG


def test_step_rejects_null_and_misaligned(zero_lib):
    Z = zero_lib
    assert _call(Z, master=None) == Z.ZERO_ERR_ARG
    assert _call(Z, grads=[6 * GB, None, 7 * GB, 8 * GB]) == Z.ZERO_ERR_ARG
    assert _call(Z, m=2 * GB + 8) == Z.ZERO_ERR_ALIGN
    assert _call(Z, grads=[6 * GB + 2, 7 * GB, 8 * GB, 9 * GB]) == Z.ZERO_ERR_ALIGN


def test_step_rejects_bad_workspace(zero_lib):
    Z = zero_lib
    assert _call(Z, ws=None) == Z.ZERO_ERR_WORKSPACE
    assert _call(Z, ws_bytes=100) == Z.ZERO_ERR_WORKSPACE
    assert _call(Z, ws=5 * GB + 16) == Z.ZERO_ERR_WORKSPACE     # not 256-byte aligned
    hp = Z.make_hparams(skip_on_overflow=True)                   # needs the FP32 copy in place
    small = Z.ZERO_WORKSPACE_CONTROL_BYTES                        # enough for the one-pass step
    assert _call(Z, hp=hp, ws_bytes=small) == Z.ZERO_ERR_WORKSPACE
    assert _call(Z, hp=hp, ws_bytes=small + 4 * 4 * 128 * 4 - 8) == Z.ZERO_ERR_WORKSPACE


def test_step_rejects_overlap(zero_lib):
    Z = zero_lib
    assert _call(Z, m=1 * GB + 256) == Z.ZERO_ERR_OVERLAP          # m inside master
    assert _call(Z, ws=4 * GB) == Z.ZERO_ERR_OVERLAP               # workspace on the weights
    assert _call(Z, grads=[6 * GB, 6 * GB, 6 * GB, 3 * GB]) == Z.ZERO_ERR_OVERLAP  # grad on v
    # read-only gradients may share memory: that passes validation and only then
    # fails on this host without a GPU, or succeeds on a GPU -- so not tested here


def test_step_into_rejects_aliasing(zero_lib):
    Z = zero_lib
    hp = Z.make_hparams(skip_on_overflow=True)
    ws_bytes = Z.zero_workspace_bytes(512, hp, False)
    g = [6 * GB]
    rc = Z.zero_step_into(g, 0, 1 * GB, 2 * GB, 3 * GB, 4 * GB, 1 * GB, 8 * GB, 9 * GB, 10 * GB,
                          128, 1, hp, 1.0, 11 * GB, ws_bytes, None, 0)
    assert rc == Z.ZERO_ERR_OVERLAP
    rc = Z.zero_step_into(g, 0, 1 * GB, 2 * GB, 3 * GB, 4 * GB, 7 * GB, 2 * GB + 64, 9 * GB,
                          10 * GB, 128, 1, hp, 1.0, 11 * GB, ws_bytes, None, 0)
    assert rc == Z.ZERO_ERR_OVERLAP
    rc = Z.zero_step_into(g, 0, 1 * GB, 2 * GB, 3 * GB, None, 7 * GB, 8 * GB, 9 * GB,
                          10 * GB, 128, 1, hp, 1.0, 11 * GB, ws_bytes, None, 0)
    assert rc == Z.ZERO_ERR_ARG   # a skipped out-of-place step needs src_w


def test_loss_scaler_matches_oracle_policy(oracle_mod):
    from zero_sharded_mixed_04_gb300.optim import LossScaler
    rng = np.random.default_rng(0)
    flags = (rng.random(200) < 0.1).tolist()
    ours = LossScaler(65536.0, True, interval=7)
    scale, good = 65536.0, 0
    for f in flags:
        ours.update(f)
        scale, good = oracle_mod.loss_scale_update(scale, good, f, 7, 0.5, 2.0)
        assert (ours.scale, ours.good_steps) == (scale, good)
    static = LossScaler(8.0, False)
    static.update(True)
    assert static.scale == 8.0


def test_constants_match_the_header(zero_lib, tmp_path):
    """Every integer #define and enum value of include/zero_gb300.h has the
    binding's value (checked against a program gcc compiles from the header)."""
    import re
    import subprocess
    header = open(os.path.join(ROOT, "include", "zero_gb300.h")).read()
    names = [n for n in re.findall(r"^#define (ZERO\w+) \S", header, re.M)]
    names += re.findall(r"^\s+(ZERO_(?:OK|STEP_\w+|ERR_\w+|GRAD_\w+))\s*=", header, re.M)
    assert {"ZERO_MAX_ELEMS", "ZERO_OK", "ZERO_ERR_BOUNDS", "ZERO_GRAD_FP32",
            "ZERO_NOALLOC_SCRATCH_BYTES"} <= set(names)
    src = tmp_path / "consts.c"
    src.write_text("\n".join(["#include <stdio.h>", '#include "zero_gb300.h"', "int main(void) {"] +
                             [f'printf("{n} %lld\\n", (long long)({n}));' for n in names] +
                             ["return 0; }"]))
    exe = tmp_path / "consts"
    subprocess.run(["gcc", "-std=c11", f"-I{os.path.join(ROOT, 'include')}", str(src), "-o",
                    str(exe)], check=True)
    out = dict(line.split() for line in subprocess.run(
        [str(exe)], check=True, capture_output=True, text=True).stdout.splitlines())
    for n in names:
        assert hasattr(zero_lib, n), f"the binding has no {n}"
        assert int(out[n]) == getattr(zero_lib, n), n


def test_struct_layouts_match_the_header(zero_lib, tmp_path):
    """The ctypes mirrors of the header's structs have the C sizes and offsets
    (checked against a program gcc compiles from include/zero_gb300.h)."""
    import subprocess
    src = tmp_path / "layout.c"
    structs = {"zero_layout": zero_lib.zero_layout, "zero_adam_hparams": zero_lib.zero_adam_hparams,
               "zero_step_result": zero_lib.zero_step_result, "zero_plan": zero_lib.zero_plan,
               "zero_device_policy": zero_lib.zero_device_policy}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "zero_gb300.h"',
             "int main(void) {"]
    for name, cls in structs.items():
        lines.append(f'printf("{name} %zu\\n", sizeof({name}));')
        for field, _ in cls._fields_:
            lines.append(f'printf("{name}.{field} %zu\\n", offsetof({name}, {field}));')
    lines += ["return 0; }"]
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", f"-I{os.path.join(ROOT, 'include')}", str(src), "-o",
                    str(exe)], check=True)
    out = dict(line.rsplit(" ", 1) for line in subprocess.run(
        [str(exe)], check=True, capture_output=True, text=True).stdout.split("\n") if line)
    for name, cls in structs.items():
        assert int(out[name]) == ctypes.sizeof(cls), name
        for field, _ in cls._fields_:
            assert int(out[f"{name}.{field}"]) == getattr(cls, field).offset, f"{name}.{field}"


def test_plan_rejects_misuse(zero_lib):
    Z = zero_lib
    hp = Z.make_hparams()
    plan = Z.zero_plan()
    n = 4 * 128 * 4
    ws_bytes = Z.zero_workspace_bytes(n, hp, True)
    rc = Z.zero_plan_init(plan, [6 * GB, 7 * GB, 8 * GB, 9 * GB], 0, 1 * GB, 2 * GB, 3 * GB, 4 * GB,
                          1 * GB, 2 * GB, 3 * GB, 4 * GB, n, 4, hp, 1.0, 5 * GB, ws_bytes)
    assert rc == Z.ZERO_OK and plan.state == 1 and plan.in_place == 1 and plan.two_pass == 0
    # a bucket before begin, and an end before all buckets, are refused on the host
    assert Z.zero_plan_bucket(plan, 0, n, None, 0) == Z.ZERO_ERR_ARG
    assert Z.zero_plan_end(plan, None, 0) == Z.ZERO_ERR_ARG
    bad = Z.zero_plan()
    assert Z.zero_plan_begin(bad, 0) == Z.ZERO_ERR_ARG
    # a plan for an out-of-place step with skip needs src_w
    hp_skip = Z.make_hparams(skip_on_overflow=True)
    rc = Z.zero_plan_init(plan, [6 * GB], 0, 1 * GB, 2 * GB, 3 * GB, None, 10 * GB, 11 * GB,
                          12 * GB, 13 * GB, 128, 1, hp_skip, 1.0, 5 * GB,
                          Z.zero_workspace_bytes(128, hp_skip, False))
    assert rc == Z.ZERO_ERR_ARG


def test_accumulation_rules(zero_lib):
    Z = zero_lib
    hp = Z.make_hparams(micro_batches=3)
    n = 4 * 128 * 4
    # accumulating needs the FP32 accumulator, in place or not
    base = Z.zero_workspace_bytes(n, Z.make_hparams(), True)
    assert Z.zero_workspace_bytes(n, hp, True) == base + 4 * n
    assert Z.zero_workspace_bytes(n, hp, False) == base + 4 * n
    # zero_step takes one batch only
    assert _call(Z, hp=hp, ws_bytes=1 << 30) == Z.ZERO_ERR_ARG
    # a plan for 3 micro-batches cannot end after covering the vector once
    plan = Z.zero_plan()
    rc = Z.zero_plan_init(plan, [6 * GB, 7 * GB, 8 * GB, 9 * GB], 0, 1 * GB, 2 * GB, 3 * GB, 4 * GB,
                          1 * GB, 2 * GB, 3 * GB, 4 * GB, n, 4, hp, 1.0, 5 * GB,
                          Z.zero_workspace_bytes(n, hp, True))
    # no clip and no in-place skip: the last micro-batch is applied in its own pass
    assert rc == Z.ZERO_OK and plan.two_pass == 0
    plan.state = 2            # as if begun, without touching a device
    plan.cursor = n
    plan.micro_batch = 0
    assert Z.zero_plan_end(plan, None, 0) == Z.ZERO_ERR_ARG
    plan.micro_batch = 1
    assert Z.zero_plan_end(plan, None, 0) == Z.ZERO_ERR_ARG
    # the update waits for the step-wide decision with clip or an in-place skip
    for kw, in_place, two in [({"max_grad_norm": 1.0}, False, 1),
                              ({"skip_on_overflow": True}, True, 1),
                              ({"skip_on_overflow": True}, False, 0)]:
        hp2 = Z.make_hparams(micro_batches=3, **kw)
        dst = [1 * GB, 2 * GB, 3 * GB, 4 * GB] if in_place else [10 * GB, 11 * GB, 12 * GB, 13 * GB]
        p2 = Z.zero_plan()
        assert Z.zero_plan_init(p2, [6 * GB, 7 * GB, 8 * GB, 9 * GB], 0, 1 * GB, 2 * GB, 3 * GB,
                                4 * GB, *dst, n, 4, hp2, 1.0, 5 * GB,
                                Z.zero_workspace_bytes(n, hp2, in_place)) == Z.ZERO_OK
        assert p2.two_pass == two, kw


@pytest.mark.parametrize("extra_rows,slack", [(0, 0), (0, 16639), (1, 0), (3, 0), (3, 16383),
                                               (63, 0), (64, 0), (65, 0), (2048, 0), (2049, 0)])
def test_plan_takes_the_rows_the_workspace_holds(zero_lib, extra_rows, slack):
    """Whatever the workspace holds beyond what the step needs becomes rows of
    norm partials: exactly as many as fit (at most 2048), none if less than
    one fits."""
    Z = zero_lib
    hp = Z.make_hparams()
    n = 4 * 128 * 4
    base = Z.ZERO_WORKSPACE_CONTROL_BYTES
    plan = Z.zero_plan()
    rc = Z.zero_plan_init(plan, [6 * GB, 7 * GB, 8 * GB, 9 * GB], 0, 1 * GB, 2 * GB, 3 * GB, 4 * GB,
                          1 * GB, 2 * GB, 3 * GB, 4 * GB, n, 4, hp, 1.0, 5 * GB,
                          base + _rows_area(extra_rows) + slack)
    assert rc == Z.ZERO_OK
    assert plan.rows_offset == base
    assert plan.row_capacity == min(extra_rows, 2048) and plan.rows_used == 0


@pytest.mark.parametrize("layers", [[5, 9, 3, 9], [100], [], [1000, 1, 1, 999], [38_597_376, 7_082_496]])
@pytest.mark.parametrize("N", [1, 4, 8])
def test_zero3_peak_matches_oracle(zero_lib, oracle_mod, layers, N):
    assert zero_lib.zero3_peak_bytes(layers, N) == oracle_mod.zero3_peak_bytes(layers, N)
    assert zero_lib.zero3_peak_bytes(layers, N, 4, 12) == oracle_mod.zero3_peak_bytes(layers, N, 4, 12)


def test_zero3_gather_rejects_bad_arguments(zero_lib):
    Z = zero_lib
    shards = [1 * GB, 2 * GB, 3 * GB, 4 * GB]
    assert Z.zero3_gather(shards, 4, 1024, 0, 4097, 5 * GB, 0) == Z.ZERO_ERR_ARG   # past the end
    assert Z.zero3_gather(shards, 4, 1020, 0, 16, 5 * GB, 0) == Z.ZERO_ERR_ARG     # shard % 8
    assert Z.zero3_gather(shards, 4, 1024, 10, 5, 5 * GB, 0) == Z.ZERO_ERR_ARG     # end < begin
    assert Z.zero3_gather(shards, 0, 1024, 0, 0, 5 * GB, 0) == Z.ZERO_ERR_ARG
    assert Z.zero3_gather(shards, 4, 1024, 0, 16, 5 * GB + 2, 0) == Z.ZERO_ERR_ALIGN
    assert Z.zero3_gather([1 * GB + 8, 2 * GB, 3 * GB, 4 * GB], 4, 1024, 0, 16, 5 * GB, 0) == \
        Z.ZERO_ERR_ALIGN
    assert Z.zero3_gather(shards, 4, 1024, 0, 16, 2 * GB + 64, 0) == Z.ZERO_ERR_OVERLAP
    assert Z.zero3_gather(shards, 4, 1024, 7, 7, None, 0) == Z.ZERO_OK              # empty: nothing
    assert Z.zero3_gather(shards, 4, 1024, 0, 16, 5 * GB, 0, flags=2) == Z.ZERO_ERR_ARG  # unknown flag


def _noalloc(Z, N=4, psi_pad=4 * 128 * 4, hp=None, dtype=None, master=1 * GB):
    hp = hp or Z.make_hparams()
    grads = [6 * GB + i * GB // 4 for i in range(N)]
    return Z.zero_step_noalloc(grads, Z.ZERO_GRAD_BF16 if dtype is None else dtype, master,
                               2 * GB, 3 * GB, 4 * GB, psi_pad, N, hp, 1.0, None, 0)


def test_noalloc_argument_errors_come_before_the_size_check(zero_lib):
    """zero_step_noalloc rejects what zero_step rejects with zero_step's code,
    whatever the size; only a call that passes those checks is held against
    the fixed array.  Fake addresses: nothing here reaches the GPU."""
    Z = zero_lib
    big = Z.ZERO_NOALLOC_MAX_TWO_PASS_ELEMS + 4 * 128   # too large for the two-pass form
    two_pass = Z.make_hparams(skip_on_overflow=True)
    assert _noalloc(Z, psi_pad=big, hp=two_pass) == Z.ZERO_ERR_TOO_LARGE
    assert _noalloc(Z, psi_pad=big + 8, hp=two_pass) == Z.ZERO_ERR_ARG       # not a multiple of N*128
    assert _noalloc(Z, psi_pad=big, hp=Z.make_hparams(skip_on_overflow=True, micro_batches=2)) \
        == Z.ZERO_ERR_ARG                                                    # one batch only
    assert _noalloc(Z, N=0, psi_pad=big, hp=two_pass) == Z.ZERO_ERR_ARG
    assert _noalloc(Z, psi_pad=big, hp=two_pass, dtype=9) == Z.ZERO_ERR_ARG
    assert _noalloc(Z, psi_pad=big, hp=Z.make_hparams(skip_on_overflow=True, lr=-1.0)) \
        == Z.ZERO_ERR_ARG
    assert _noalloc(Z, psi_pad=big, hp=two_pass, master=None) == Z.ZERO_ERR_ARG
    assert _noalloc(Z, psi_pad=big, hp=two_pass, master=1 * GB + 4) == Z.ZERO_ERR_ALIGN


def test_pingpong_argument_checks(zero_lib):
    """zero_plan_set_pingpong wants an initialised out-of-place plan whose two
    sets are complete and disjoint.  Fake addresses: every call here is
    rejected before any CUDA call."""
    torch = pytest.importorskip("torch")
    Z = zero_lib
    N, n = 4, 4 * 128 * 4
    grads = [6 * GB + i * GB // 4 for i in range(N)]
    hp = Z.make_hparams(skip_on_overflow=True)
    ws = 5 * GB
    wsb = Z.zero_workspace_bytes(n, hp, False)
    word = 11 * GB

    def plan_of(src, dst, state=None):
        plan = Z.zero_plan()
        rc = Z.zero_plan_init(plan, grads, Z.ZERO_GRAD_BF16, *src, *dst, n, N, hp, 1.0, ws, wsb)
        assert rc == Z.ZERO_OK
        return plan

    src = [1 * GB, 2 * GB, 3 * GB, 4 * GB]
    dst = [12 * GB, 13 * GB, 14 * GB, 15 * GB]
    plan = Z.zero_plan()
    assert Z.zero_plan_set_pingpong(plan, word) == Z.ZERO_ERR_ARG          # not initialised
    p_in = Z.zero_plan()
    assert Z.zero_plan_init(p_in, grads, Z.ZERO_GRAD_BF16, *src, *src, n, N,
                            Z.make_hparams(), 1.0, ws,
                            Z.zero_workspace_bytes(n, Z.make_hparams(), True)) == Z.ZERO_OK
    assert Z.zero_plan_set_pingpong(p_in, word) == Z.ZERO_ERR_ARG          # in place
    p = plan_of(src, dst)
    assert Z.zero_plan_set_pingpong(p, None) == Z.ZERO_ERR_ARG
    assert Z.zero_plan_set_pingpong(p, word + 2) == Z.ZERO_ERR_ARG         # misaligned
    # a src buffer that overlaps a gradient is fine while src is only read,
    # not once ping-pong makes it an output too
    p = plan_of([grads[1], 2 * GB, 3 * GB, 4 * GB], dst)
    assert Z.zero_plan_set_pingpong(p, word) == Z.ZERO_ERR_OVERLAP


def test_release_build_has_no_bounds_checks(zero_lib):
    """The release library reports -1 (no checks compiled in) without any CUDA
    call; the debug library exports the same entry points."""
    import ctypes as C
    from zero_sharded_mixed_04_gb300 import build
    if zero_lib.DEBUG_BUILD:
        pytest.skip("the binding loaded the debug build")
    assert zero_lib.zero_debug_bounds_violations() == -1
    if os.path.exists(build.DEBUG_LIB_PATH):
        dbg = C.CDLL(build.DEBUG_LIB_PATH)
        for name in _declared_functions():
            assert hasattr(dbg, name), f"{name} missing from the debug build"


@pytest.mark.parametrize("which", ["ragged6b", "gpt2small"])
@pytest.mark.parametrize("N", [4, 8])
def test_layout_of_the_workload_tensor_lists(zero_lib, oracle_mod, which, N):
    """The C-ABI layout of the workloads' own tensor lists: the ragged
    6,000,000,007-parameter list (about 90 tensors of 1 to 2^27 elements) and
    GPT-2-small's, against the oracle's layout, offsets and shard ranges."""
    from zero_sharded_mixed_04_gb300 import synth
    sizes = (synth.ragged6b_tensor_sizes() if which == "ragged6b"
             else synth.gpt2_small_tensor_sizes())
    rc, lay, offs = zero_lib.zero_init_layout(sizes, N)
    assert rc == zero_lib.ZERO_OK
    o_offs, psi, psi_pad, shard = oracle_mod.layout(sizes, N)
    assert (lay.psi, lay.psi_pad, lay.shard, lay.n_tensors) == (psi, psi_pad, shard, len(sizes))
    assert list(offs) == list(o_offs)
    if which == "ragged6b":
        assert psi == 6_000_000_007 and 1 in sizes and (1 << 27) in sizes
        assert psi_pad % (N * 128) == 0 and psi_pad - psi < N * 128
    else:
        assert psi == 123_588_864
    for r in range(N):
        rc, b, e = zero_lib.zero_shard_range(lay, r)
        assert rc == 0 and (b, e) == (r * shard, (r + 1) * shard)



def _rows_area(rows):
    """Bytes of the rows of norm partials for `rows` launches: the carry,
    padded to 256 bytes, then 2048 FP64 slots per row."""
    if rows <= 0:
        return 0
    return 256 + rows * 2048 * 8


def _launches(psi_pad, bucket):
    """Launches of one pass: each bucket in near-equal parts of at most 2^22 elements."""
    def parts(n):
        return 0 if n <= 0 else -(-n // (1 << 22))
    bucket = bucket or psi_pad
    full = psi_pad // bucket
    return min(2048, full * parts(bucket) + parts(psi_pad - full * bucket))


@pytest.mark.parametrize("psi_pad,bucket,skip,in_place", [
    (4 * 128 * 4, 0, False, True),                 # one launch
    (1_000_000_512, 25_000_000, True, False),      # flat1b_n8: 40 buckets x 6 launches + 1
    (123_589_120, 0, False, True),                 # gpt2small_n4: 30 launches
    (6_000_000_512, 0, False, True),               # ragged6b_n4: 1431 launches
    (3_000_000_000, 0, True, True),                # two-pass: the FP32 gradient first
    (1 << 20, 8, False, True),                     # tiny buckets: capped at 2048 rows
])
def test_workspace_bytes_include_rows_of_partials(zero_lib, psi_pad, bucket, skip, in_place):
    """zero_workspace_bytes = the part every step needs (control block and
    shared slots, plus the FP32 combined gradient of the two-pass form), then
    one row of norm partials per first-pass launch of the step."""
    Z = zero_lib
    hp = Z.make_hparams(skip_on_overflow=skip, bucket_elems=bucket)
    need = Z.ZERO_WORKSPACE_CONTROL_BYTES + (4 * psi_pad if (skip and in_place) else 0)
    want = -(-need // 256) * 256 + _rows_area(_launches(psi_pad, bucket))
    assert Z.zero_workspace_bytes(psi_pad, hp, in_place) == want
    if psi_pad == 1_000_000_512:
        assert _launches(psi_pad, bucket) == 241
    if psi_pad == 6_000_000_512:
        assert _launches(psi_pad, bucket) == 1431


def test_binding_pads_a_short_gradient_list(zero_lib):
    """Fewer gradient pointers than N reach the library as NULLs, an argument
    error, never as a read past the end of the pointer array."""
    Z = zero_lib
    hp = Z.make_hparams()
    n = 4 * 128 * 4
    ws = Z.zero_workspace_bytes(n, hp, True)
    rc = Z.zero_step([6 * GB, 7 * GB, 8 * GB], Z.ZERO_GRAD_BF16, 1 * GB, 2 * GB, 3 * GB, 4 * GB,
                     n, 4, hp, 1.0, 5 * GB, ws, None, 0)
    assert rc == Z.ZERO_ERR_ARG
    # a plan may take its gradients per bucket: the missing ranks stay NULL
    plan = Z.zero_plan()
    assert Z.zero_plan_init(plan, [6 * GB], Z.ZERO_GRAD_BF16, 1 * GB, 2 * GB, 3 * GB, 4 * GB,
                            1 * GB, 2 * GB, 3 * GB, 4 * GB, n, 4, hp, 1.0, 5 * GB, ws) == 0
    assert plan.grads[0] == 6 * GB and not any(plan.grads[1:4])
    assert Z.zero3_gather([6 * GB], 4, 1024, 0, 8, 5 * GB, 0, 0) == Z.ZERO_ERR_ARG


def test_binding_refuses_tensors_too_small_for_the_call(zero_lib):
    """Torch tensors passed as buffers must hold what the call touches and be
    contiguous; the binding refuses them before the library sees a pointer."""
    torch = pytest.importorskip("torch")
    Z = zero_lib
    N, n = 4, 4 * 128 * 4
    hp = Z.make_hparams()
    ws = torch.empty(Z.zero_workspace_bytes(n, hp, True), dtype=torch.uint8)
    grads = [torch.zeros(n, dtype=torch.bfloat16) for _ in range(N)]
    st = [torch.zeros(n), torch.zeros(n), torch.zeros(n), torch.zeros(n, dtype=torch.int16)]

    def call(g=grads, s=st, w=ws, wsb=ws.numel(), dtype=Z.ZERO_GRAD_BF16):
        return Z.zero_step(g, dtype, *s, n, N, hp, 1.0, w, wsb, None, 0)

    with pytest.raises(ValueError, match=r"grads\[2\]"):
        call(g=grads[:2] + [torch.zeros(n - 8, dtype=torch.bfloat16)] + grads[3:])
    with pytest.raises(ValueError, match=r"grads\[0\]"):   # FP32 gradients need 4 bytes each
        call(dtype=Z.ZERO_GRAD_FP32)
    with pytest.raises(ValueError, match="w_bf16"):
        call(s=st[:3] + [torch.zeros(n // 2, dtype=torch.int16)])
    with pytest.raises(ValueError, match="not contiguous"):
        call(s=[torch.zeros(2 * n)[::2]] + st[1:])
    with pytest.raises(ValueError, match="workspace"):
        call(wsb=ws.numel() + 1)
    with pytest.raises(ValueError, match="view"):
        Z.zero3_gather([torch.zeros(1024, dtype=torch.int16)] * N, N, 1024, 0, 2048,
                       torch.zeros(1024, dtype=torch.int16), 0, 0)
    plan = Z.zero_plan()
    plan.grad_dtype, plan.N, plan.psi_pad = Z.ZERO_GRAD_BF16, N, n
    with pytest.raises(ValueError, match=r"bucket_grads\[1\]"):
        Z.zero_plan_bucket(plan, 0, 512, [torch.zeros(512, dtype=torch.bfloat16),
                                          torch.zeros(256, dtype=torch.bfloat16)], 0)
    # a size the library refuses is left for it to refuse, whatever the buffers hold
    small = torch.zeros(8, dtype=torch.int16)
    assert Z.zero3_gather([small] * N, N, 1024, 0, 4097, small, 0, 0) == Z.ZERO_ERR_ARG
    assert Z.zero_plan_bucket(plan, 0, n + 512, [small] * N, 0) == Z.ZERO_ERR_ARG


@pytest.mark.parametrize("lr,beta1,beta2", [(1e-3, 0.9, 0.999), (3e-4, 0.8, 0.95),
                                            (1e-2, 0.0, 0.0), (0.1, 0.999, 0.99999)])
def test_policy_table_matches_the_oracle_scalars(zero_lib, oracle_mod, lr, beta1, beta2):
    """Every entry of a device-policy table is the oracle's FP32 step_size and
    sqrt(1 - beta2^t) for its t, bit for bit, from t = 1 into the range where
    the bias corrections reach 1, and across 2^31 (t is 64-bit on both sides)."""
    Z = zero_lib
    hp = Z.make_hparams(lr=lr, beta1=beta1, beta2=beta2, step=7)
    ohp = oracle_mod.Hparams(lr=lr, beta1=beta1, beta2=beta2)
    for t_first, t_count in ((1, 300), (999_990, 20), ((1 << 31) - 4, 8), (1 << 40, 3)):
        table = (ctypes.c_float * (2 * t_count))()
        assert Z.zero_policy_table_fill(hp, t_first, t_count, ctypes.addressof(table)) == Z.ZERO_OK
        for i in range(t_count):
            s = oracle_mod.step_scalars(ohp, t_first + i, 4, 1.0)
            want = np.array([s["step_size"], s["sbc2"]], np.float32)
            got = np.array([table[2 * i], table[2 * i + 1]], np.float32)
            assert got.tobytes() == want.tobytes(), (t_first + i, got, want)
    assert hp.step == 7  # the caller's hyper-parameters are left alone


def test_policy_table_rejects_bad_arguments(zero_lib):
    Z = zero_lib
    hp = Z.make_hparams()
    table = (ctypes.c_float * 8)()
    a = ctypes.addressof(table)
    for t_first, t_count in ((0, 1), (1, 0), (-5, 2), (1, -1), (Z.ZERO_MAX_ELEMS, 2),
                             (2, Z.ZERO_MAX_ELEMS)):
        assert Z.zero_policy_table_fill(hp, t_first, t_count, a) == Z.ZERO_ERR_ARG
    assert Z.zero_policy_table_fill(hp, 1, 1, None) == Z.ZERO_ERR_ARG
    assert Z.zero_policy_table_fill(Z.make_hparams(beta2=1.0), 1, 1, a) == Z.ZERO_ERR_ARG
    assert list(table) == [0.0] * 8
    assert Z.zero_policy_table_fill(hp, Z.ZERO_MAX_ELEMS, 1, a) == Z.ZERO_OK
    # a plan that has not been initialised takes no table
    plan = Z.zero_plan()
    assert Z.zero_plan_set_device_policy_table(plan, a, a, 1, 4) == Z.ZERO_ERR_ARG
