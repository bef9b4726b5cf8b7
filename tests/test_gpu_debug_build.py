"""The debug build (libzero_gb300_debug.so, the same sources compiled with
-DZERO_DEBUG) on the GPU.  Its kernels check every index range against the
lengths of the buffers before touching it; nothing traps.

* parity: correct runs of every kernel form match the oracle and the checks
  find nothing;
* sweep: the same for 128 configurations of the random parity sweep;
* overrun: launches made to run past the end of the buffers (a debug-only
  test setting) have every out-of-range access skipped and counted, end with
  ZERO_ERR_BOUNDS, and leave the guard regions behind every buffer as they
  were.  The guard regions are larger than the overrun, so an access a check
  missed would still stay inside this process's own allocations.

Each case runs in a child process, which loads the debug library instead of
the release one.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def _run(case, extra_env=None):
    env = dict(os.environ, ZERO_GB300_DEBUG="1")
    env.pop("ZERO_DEBUG_TEST_OVERRUN", None)
    env.update(extra_env or {})
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_build_cases.py"), case],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-3000:]
    return r.stdout


def test_debug_build_parity(zero_lib):
    assert "debug build parity: ok" in _run("parity")


def test_debug_build_random_sweep(zero_lib):
    assert "debug build sweep: ok" in _run("sweep")


def test_debug_build_skips_out_of_range_accesses(zero_lib):
    assert "debug build overrun: ok" in _run("overrun", {"ZERO_DEBUG_TEST_OVERRUN": "64"})
