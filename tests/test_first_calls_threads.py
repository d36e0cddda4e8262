"""The library's one-time per-device set-up (kernel shared-memory limits, the
pair kernels' cluster occupancy, the device's cached properties) is reached
first by several host threads at once, in a fresh process: every product
still runs and meets its bound (first_calls_worker.py)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_first_calls_from_several_threads_at_once():
    r = subprocess.run([sys.executable, os.path.join(HERE, "first_calls_worker.py")],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, (r.stdout[-3000:], r.stderr[-3000:])
    assert r.stdout.count("worst") == 8
