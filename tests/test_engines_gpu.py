"""Every op on each engine choice (MGSCAN_ENGINE=chunked / stream), against
the oracle.  The library reads the variable once per process, so each choice
runs engine_check.py in a child process of its own."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("engine", ["chunked", "stream"])
def test_engine_parity(cuda_lib, engine):
    env = dict(os.environ, MGSCAN_ENGINE=engine)
    r = subprocess.run([sys.executable, os.path.join(HERE, "engine_check.py")], env=env,
                       capture_output=True, text=True, timeout=600)
    print(r.stdout)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
