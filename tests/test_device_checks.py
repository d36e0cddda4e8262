"""The build with device-side bounds checks (python -m dense_gemm_14_gb300.build
--checked; csrc/checks.h): every plain global store of C and every stream-K
slot and flag access is tested against its buffer's bounds before it
happens. Run over every kernel, loader and schedule (device_checks_worker.py,
in a subprocess that loads the checked library through GEMM14_LIB), no check
may fail, and the results must be the product build's bit for bit: the
checks change no arithmetic."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import dense_gemm_14_gb300 as g14
from dense_gemm_14_gb300 import build

import device_checks_worker as worker

pytestmark = pytest.mark.gpu


def test_checked_build_passes_and_matches_the_product(tmp_path):
    lib = build.build(checked=True)
    assert os.path.abspath(lib) != os.path.abspath(g14.lib_path())
    out = tmp_path / "checked.npz"
    env = dict(os.environ, GEMM14_LIB=lib)
    r = subprocess.run([sys.executable, worker.__file__, str(out)], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    got = np.load(out)
    assert str(got["lib"]) == lib
    stream = torch.cuda.current_stream().cuda_stream
    for i, case in enumerate(worker.CASES):
        st = int(got[f"s{i}"])
        assert st == 0, (case[0], g14.status_string(st))
        want, st_product = worker.run_case(case, stream)
        assert st_product == 0, case[0]
        assert not np.isnan(want[:, :case[5]]).any(), case[0]
        assert np.array_equal(got[f"c{i}"], want, equal_nan=True), case[0]
