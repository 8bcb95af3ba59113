"""The parity tests again, against the bounds-check build of the library.

A memory sanitizer is not available on this device's pool.  Its substitute:
build() also makes libmoe_decode_bounds.so, the same sources compiled with
MOE_BOUNDS_CHECK, in which every index that comes from data (a pair id, a
pooled position, a routed row) is tested before it addresses memory and a bad
one latches device error 3 instead of faulting; and every handle's workspace
regions are followed by guards that each error check verifies.  This runs the
GPU parity tests (all but the full-size end-to-end ones, which run against
the default build) in a child process that loads the bounds-check library;
every test there checks the handle's error word, so an index out of range
anywhere fails it.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_parity_under_the_bounds_check_build():
    from speculative_decode_routed_gb300 import _build as pb
    assert os.path.exists(pb.LIB_BOUNDS), "build() makes the bounds-check library"
    env = dict(os.environ, MOE_DECODE_LIB=pb.LIB_BOUNDS, MOE_DECODE_EXPECT_BOUNDS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_gpu_parity.py", "-m", "gpu", "-q",
                        "-p", "no:cacheprovider", "-k", "not end_to_end or tiny"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    tail = r.stdout[-4000:] + r.stderr[-2000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and "failed" not in r.stdout, tail
