"""The debug-bounds build (-DMOE_DEBUG_BOUNDS) stands in for compute-sanitizer,
which is closed on this machine: its kernels check every index they read back from
a routing buffer (block count against the capacity, expert ids, pair ids)
before use and record MOE_DEVERR_BOUNDS instead of going out of range.  On valid
inputs no check may fire and the results must still match the oracle.  The
library is chosen once per process, so the cases run in a child process."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_debug_bounds_build_is_clean_and_matches_the_oracle():
    env = dict(os.environ, MOE_INT4_DEBUG_BOUNDS="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_bounds_check.py")], env=env,
                       capture_output=True, text=True, timeout=600)
    print(r.stdout)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "debug-bounds: all cases clean" in r.stdout
