"""The small-case GPU parity suites again, on the bounds-checking build of the library.

That build (GDN_DEBUG_BOUNDS) checks every global copy source and every store
of the decode, replay, speculative-step, prefill and rollback kernels against
the extent of its array; an access outside is skipped and sets
GDN_DEVERR_BOUNDS in the error word, never a fault. The parity tests assert a
clear error word after every call, so a passing run shows that no index of
those kernels leaves its array on these cases -- multi-round grids with
ragged tails, rings that wrap and fold, windows at the largest ring and head,
padding and out-of-range slots. The replay tests also keep poisoned canary
bytes around every cache array and output, checked bit-exactly after each
call (tests/gpu_util.py: guarded).

The suites run in a child process that loads the bounds-checking library
through GDN_LIBRARY.
"""
import os
import subprocess
import sys

import pytest

from hybrid_ssm_gated_gb300 import build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITES = ["tests/test_gpu_decode.py", "tests/test_gpu_replay.py", "tests/test_gpu_mamba2.py", "tests/test_gpu_spec.py",
          "tests/test_gpu_prefill.py"]


def test_small_suites_on_the_bounds_checking_build():
    lib = build.build(debug=True)
    env = dict(os.environ, GDN_LIBRARY=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu and not slow", "-p", "no:cacheprovider"]
                       + SUITES, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
