"""The pins catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of oracle/zero_oracle.c, builds it, and
runs the fast pin tests against that build in a fresh process: they must
fail.  The mistakes are the kind a restatement of the method could contain.
  - A dropped term: bias correction, the 1/N of the batch mean, the last rank.
  - A wrong operator or sign: the update's sign, eps inside the square root,
    v fed g instead of g*g.
  - Swapped roles: beta1 with beta2.
  - A wrong index: a neighbour's gradient, a transposed shard index.
  - Rounding slips: BF16 truncation, ties rounded away from even.
  - Wrong step-wide rules: a skip that does not skip, a clip coefficient not
    capped at 1, weight decay without the learning rate.
  - A wrong ledger formula.
  - A wrong summation order or start: the ranks added in reverse or in
    pairs, a sum started from rank 0's value instead of +0, and the same two
    slips for the micro-batches of an accumulated step.
"""
import concurrent.futures
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "zero_oracle.c")

MUTANTS = {
    "no_bias_correction_1": ("s->step_size = (float)(hp->lr / bc1);",
                             "s->step_size = (float)(hp->lr);"),
    "eps_inside_sqrt": ("float den = sqrtf(vv) / s->sbc2 + s->eps;",
                        "float den = sqrtf(vv + s->eps) / s->sbc2;"),
    "beta_roles_swapped": ("mm = s->b1 * mm + s->omb1 * g;", "mm = s->b2 * mm + s->omb2 * g;"),
    "update_sign_flipped": ("pp = pp - s->step_size * (mm / den);",
                            "pp = pp + s->step_size * (mm / den);"),
    "no_batch_mean": ("s->inv = (float)(1.0 / ((double)N * loss_scale));",
                      "s->inv = (float)(1.0 / loss_scale);"),
    "neighbour_gradient": ("a = a + orc_load_grad(grads[i], dtype, idx);",
                           "a = a + orc_load_grad(grads[i], dtype, idx ^ 1);"),
    "last_rank_dropped": ("for (int32_t i = 0; i < N; ++i)\n        a = a + orc_load_grad",
                          "for (int32_t i = 0; i + 1 < N; ++i)\n        a = a + orc_load_grad"),
    "shard_index_transposed": ("out_shard[j] = orc_reduce_element(grads, dtype, N, (int64_t)r * shard + j, inv);",
                               "out_shard[j] = orc_reduce_element(grads, dtype, N, j * N + r, inv);"),
    "bf16_truncates": ("    if (dropped > 0x8000u)\n        kept += 1u;\n    else if",
                       "    if (0)\n        kept += 1u;\n    else if"),
    "bf16_ties_away": ("else if (dropped == 0x8000u && (kept & 1u) != 0u)",
                       "else if (dropped == 0x8000u)"),
    "decay_without_lr": ("s->decay = (float)(1.0 - hp->lr * hp->weight_decay);",
                         "s->decay = (float)(1.0 - hp->weight_decay);"),
    "skip_ignored": ("    if (skip_on_overflow && bad) {\n        res->applied = 0;\n        free(g);",
                     "    if (0) {\n        res->applied = 0;\n        free(g);"),
    "clip_not_capped": ("return (c < 1.0) ? (float)c : 1.0f;", "return (float)c;"),
    "zero2_ledger_wrong": ("return weight_bytes * psi + (grad_bytes + optim_bytes) * sharded;",
                           "return (weight_bytes + grad_bytes) * psi + optim_bytes * sharded;"),
    "v_without_square": ("vv = s->b2 * vv + s->omb2 * (g * g);", "vv = s->b2 * vv + s->omb2 * g;"),
    "gather_shard_index_transposed": ("out[j - begin] = shards[j / shard][j % shard];",
                                      "out[j - begin] = shards[j % N][j / N];"),
    "peak_forgets_prefetched_view": (
        "int64_t pair = layer_numel[i] + (i + 1 < n_layers ? layer_numel[i + 1] : 0);",
        "int64_t pair = layer_numel[i];"),
    "reduction_order_reversed": (
        "for (int32_t i = 0; i < N; ++i)\n        a = a + orc_load_grad(grads[i], dtype, idx);",
        "for (int32_t i = N - 1; i >= 0; --i)\n        a = a + orc_load_grad(grads[i], dtype, idx);"),
    "reduction_in_pairs": (
        "for (int32_t i = 0; i < N; ++i)\n        a = a + orc_load_grad(grads[i], dtype, idx);",
        "for (int32_t i = 0; i + 1 < N; i += 2)\n"
        "        a = a + (orc_load_grad(grads[i], dtype, idx) + orc_load_grad(grads[i + 1], dtype, idx));\n"
        "    if (N % 2)\n        a = a + orc_load_grad(grads[N - 1], dtype, idx);"),
    "reduction_starts_from_rank0": (
        "float a = 0.0f;\n    for (int32_t i = 0; i < N; ++i)",
        "float a = orc_load_grad(grads[0], dtype, idx);\n    for (int32_t i = 1; i < N; ++i)"),
    "micro_batches_reversed": (
        "for (int32_t mb = 0; mb < k; ++mb)",
        "for (int32_t mb = k - 1; mb >= 0; --mb)"),
    "accumulator_starts_from_first_micro_batch": (
        "        acc[j] = 0.0f;\n    for (int32_t mb = 0; mb < k; ++mb)",
        "        acc[j] = orc_reduce_element(grads, dtype, N, j, inv);\n"
        "    for (int32_t mb = 1; mb < k; ++mb)"),
    "norm_squares_in_fp32": (
        "s = s + (double)g[j] * (double)g[j];",
        "s = s + (double)(g[j] * g[j]);"),
    "accumulation_mean_without_k": (
        "float inv = (float)(1.0 / ((double)N * (double)k * loss_scale));",
        "float inv = (float)(1.0 / ((double)N * loss_scale));"),
}

PIN_TESTS = ["tests/test_oracle_adam.py", "tests/test_oracle_collectives.py",
             "tests/test_oracle_step.py", "tests/test_oracle_ledger.py",
             "tests/test_oracle_bf16.py", "tests/test_oracle_accum.py",
             "tests/test_oracle_zero3.py"]


def _build_mutant(name, tmp):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"{name}: the planted text must match the oracle exactly once"
    path_c = os.path.join(tmp, f"{name}.c")
    with open(path_c, "w") as f:
        f.write(src.replace(old, new))
    path_so = os.path.join(tmp, f"{name}.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                    "-shared", "-o", path_so, path_c, "-lm"], check=True)
    return path_so


def _pins_fail(lib):
    env = dict(os.environ, ORACLE_LIB_OVERRIDE=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "-m", "not gpu", "-k", "not every_fp32_pattern", *PIN_TESTS],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode != 0, r.stdout[-400:]


def test_unmutated_oracle_passes_its_pins(tmp_path):
    src = os.path.join(tmp_path, "same.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                    "-shared", "-o", src, SRC, "-lm"], check=True)
    failed, out = _pins_fail(src)
    assert not failed, out


def test_every_planted_mistake_fails_a_pin(tmp_path):
    libs = {name: _build_mutant(name, str(tmp_path)) for name in MUTANTS}
    with concurrent.futures.ThreadPoolExecutor(max(1, min(8, os.cpu_count() or 1))) as ex:
        results = dict(zip(libs, ex.map(_pins_fail, libs.values())))
    survivors = [name for name, (failed, _) in results.items() if not failed]
    assert not survivors, f"mistakes no pin caught: {survivors}"
