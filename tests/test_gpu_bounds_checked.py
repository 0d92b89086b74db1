"""The bounds-checked build of the library on the parity cases.

Memory checkers are not available on every GPU host, so the library can be
built with every kernel index validated in-kernel (-DLIONCUB_BOUNDS_CHECK): an
index outside its buffer sets a bit in the handle's status word and the
access is skipped.  This test builds that variant and reruns a spread of the
parity cases with it (ragged sizes, every code width, sync, ties, exact
zeros, the full 1M-element workload, guard bands, diagnostics).  The parity
harness checks the status word after every run, so any out-of-bounds index
fails the test, and the results must still match the oracle.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_parity_cases_under_bounds_checks():
    from communication_compressed_sign_gb300 import build
    import __graft_entry__
    __graft_entry__.build()
    lib = build.build(bounds_check=True)
    sel = ("small_ragged or multi_tensor or tie_and_average or exact_zero or all_layer or workload1 "
           "or guard_bands or diagnose_small or diagnose_qinf_small or host_buffer or empty_vector or many_small")
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_gpu_parity.py", "-m", "gpu", "-x", "-q",
                        "-p", "no:cacheprovider", "-k", sel],
                       cwd=ROOT, env={**os.environ, "LIONCUB_LIBRARY": lib}, capture_output=True, text=True,
                       timeout=1200)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and "failed" not in r.stdout, tail
