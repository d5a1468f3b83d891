"""A pipeline wait that runs out on the GPU: the debug-bounds build leaves one
weight stage's copy unissued (a barrier that nothing completes), and the call
must report MOE_DEVERR_TIMEOUT, return, and leave the context usable.  The
library is chosen once per process, so the cases run in a child process."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_wait_that_runs_out_is_reported_and_the_context_recovers():
    env = dict(os.environ, MOE_INT4_DEBUG_BOUNDS="1")
    env.pop("MOE_INT4_DEBUG_SKIP_STAGE", None)
    r = subprocess.run([sys.executable, os.path.join(HERE, "timeout_check.py")], env=env,
                       capture_output=True, text=True, timeout=600)
    print(r.stdout)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "timeouts: all cases reported and recovered" in r.stdout
