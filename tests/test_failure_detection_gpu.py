"""Failure detection on the GPU without a GPU fault.

Every pipelined kernel bounds its mbarrier waits; a wait that runs out sets
bit 0 of the device error word and the kernel returns. Here a diagnostic
kernel waits on an mbarrier that nothing ever completes (a short poll limit),
and the host reads the error status; the context must stay usable.
"""
import numpy as np
import pytest

from oracle import check, gate
from rmsnorm_fwd_bwd_gb300 import binding as B
from rmsnorm_fwd_bwd_gb300 import inputs

from . import gpu_util

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_instead_of_hanging():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    assert B.rmsnorm_device_error(clear=True) == 0
    assert B.rmsnorm_selftest_wait_timeout(0) == 9            # RMSNORM_ERR_ARG
    assert B.rmsnorm_selftest_wait_timeout(4096) == B.RMSNORM_OK
    torch.cuda.synchronize()
    assert B.rmsnorm_device_error(clear=True) & 1
    assert B.rmsnorm_device_error() == 0
    # the context is still usable: a normal forward/backward passes the gate
    x, g, dy = inputs.make_inputs(64, 4096, "bfloat16", seed=2)
    y, r, dx, dg = gpu_util.run(x, g, dy, "bfloat16")
    res = check.gate_outputs(x, g, dy, "bfloat16", False, 1e-6, y=y, rstd=r, dx=dx, dgamma=dg)
    assert gate.overall(res) == "PASS", gate.report("after timeout", res)
    assert B.rmsnorm_device_error() == 0


def test_autograd_surfaces_the_device_error_word(monkeypatch):
    """The torch ops succeed on the host even when a kernel gave up a bounded
    wait; check_device_error (or RMSNORM_CHECK_DEVICE_ERROR=1, every op) turns
    the device error word into an exception. The word is set by the diagnostic
    wait kernel, never by a fault."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rmsnorm_fwd_bwd_gb300 import autograd as ag
    B.rmsnorm_device_error(clear=True)
    x = torch.randn(16, 512, device="cuda", dtype=torch.bfloat16)
    w = torch.ones(512, device="cuda", dtype=torch.bfloat16)
    ag.rms_norm(x, w)
    ag.check_device_error()                                   # clean: no exception
    assert B.rmsnorm_selftest_wait_timeout(4096) == B.RMSNORM_OK
    with pytest.raises(ag.DeviceError):
        ag.check_device_error()
    ag.check_device_error()                                   # the check cleared the word
    monkeypatch.setattr(ag, "CHECK_EVERY_OP", True)
    assert B.rmsnorm_selftest_wait_timeout(4096) == B.RMSNORM_OK
    with pytest.raises(ag.DeviceError):
        ag.rms_norm(x, w)
    assert B.rmsnorm_device_error(clear=True) == 0
