"""The debug build of the library (-DRMSNORM_DEBUG) on the GPU: its kernels
check every TMA read against the extent of the tensor read and report a read
outside it through bit 1 of the device error word. Runs the cases of
tests/debug_build_cases.py in a child process that loads the debug build
(RMSNORM_LIBRARY) and requires gated results and a clear error word."""
import os
import subprocess
import sys

import pytest

from rmsnorm_fwd_bwd_gb300 import build as build_mod

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_debug_build_reads_stay_inside_their_tensors():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = build_mod.build(debug=True)
    env = dict(os.environ, RMSNORM_LIBRARY=lib)
    res = subprocess.run([sys.executable, "-m", "tests.debug_build_cases"], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=900)
    print(res.stdout[-4000:], res.stderr[-4000:])
    assert res.returncode == 0
    assert "device error word 0" in res.stdout
