"""The bounds-checked debug build (librf_gb300_dbg.so): ragged cases of
every entry point run clean against the oracle with every thread-issued
global access checked, and the checker itself reports an index past a
tensor's end.  Runs tests/bounds_debug_cases.py in a process of its own,
because the package picks its library (RF_GB300_LIB=debug) at import."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_debug_build_runs_every_path_clean():
    env = dict(os.environ, RF_GB300_LIB="debug")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "bounds_debug_cases.py")],
                       cwd=ROOT, env=env, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:]
    assert "every case clean" in r.stdout
