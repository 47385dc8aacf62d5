"""NVTX ranges (DSA_NVTX=1 in the environment): marking the entry points,
the forward's query chunks and every kernel launch for timeline tools leaves
the results unchanged.  The switch is read once per process, so the check runs
the small forward of the smoke test (which compares with the oracle) in a
child process."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_forward_with_nvtx_ranges():
    env = dict(os.environ, DSA_NVTX="1")
    r = subprocess.run([sys.executable, "-c", "import __graft_entry__ as g; g.smoke(); print('smoke ok')"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and "smoke ok" in r.stdout, (r.stdout[-2000:], r.stderr[-4000:])
