"""The C-ABI library builds, loads and exports every declared symbol (CPU only).

Only host-side validation is exercised here: each call below fails its
argument checks before the library touches CUDA, so no GPU is needed.
"""
import ctypes
import os

import pytest

from rmsnorm_fwd_bwd_gb300 import binding as B
from rmsnorm_fwd_bwd_gb300 import build as build_mod


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return ctypes.CDLL(B.LIB_PATH)


def test_header_declares_the_boundary():
    names = B.header_functions()
    for required in ("rmsnorm_fwd", "rmsnorm_bwd", "rmsnorm_bwd_workspace_size",
                     "rmsnorm_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in B.header_functions():
        assert hasattr(lib, name), name


def test_binding_has_the_same_names():
    for name in B.header_functions():
        assert callable(getattr(B, name)), name


def test_status_strings():
    for code in range(10):
        s = B.rmsnorm_status_string(code)
        assert isinstance(s, str) and s
    assert B.rmsnorm_status_string(0) == "ok"
    assert B.rmsnorm_status_string(12345) == "unknown status"


def test_host_validation_without_gpu():
    # invalid dtype, offset, shape and eps, then NULL and misaligned pointers
    assert B.rmsnorm_fwd(None, None, None, None, 4, 8, 1e-6, 5, 0, 0) == 3
    assert B.rmsnorm_fwd(None, None, None, None, 4, 8, 1e-6, 0, 3, 0) == 9
    assert B.rmsnorm_fwd(None, None, None, None, 4, 0, 1e-6, 0, 0, 0) == 2
    assert B.rmsnorm_fwd(None, None, None, None, -1, 8, 1e-6, 0, 0, 0) == 2
    assert B.rmsnorm_fwd(None, None, None, None, 4, 16385, 1e-6, 0, 0, 0) == 2
    assert B.rmsnorm_fwd(None, None, None, None, 4, 8, 0.0, 0, 0, 0) == 4
    assert B.rmsnorm_fwd(None, None, None, None, 4, 8, -1e-6, 0, 0, 0) == 4
    assert B.rmsnorm_fwd(None, None, None, None, 4, 8, float("inf"), 0, 0, 0) == 4
    assert B.rmsnorm_fwd(None, None, None, None, 4, 8, 1e-6, 0, 0, 0) == 1
    assert B.rmsnorm_fwd(0x1002, 0x2000, 0x3000, 0x4000, 4, 8, 1e-6, 0, 0, 0) == 5
    assert B.rmsnorm_bwd(None, None, None, None, None, None, 4, 8, 0, 0, None, 0, 0) == 1
    assert B.rmsnorm_bwd(None, None, None, None, None, 0x1001, 4, 8, 1, 0, None, 0, 0) == 5
    assert B.rmsnorm_bwd(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 4, 8, 2, 0,
                         0x1008, 1 << 20, 0) == 5   # workspace not 16-byte aligned
    assert B.rmsnorm_bwd_workspace_size(0, 8, 0) == 0
    assert B.rmsnorm_bwd_workspace_size(4, 0, 0) == 0
    assert B.rmsnorm_bwd_workspace_size(4, 8, 9) == 0
    assert B.rmsnorm_set_launch_override(5, 0, 0, 0, 0) == 9
    assert B.rmsnorm_set_launch_override(-1, 0, 0, 0, 0) == 9
    assert B.rmsnorm_set_launch_override(3, 0, 0, 0, 0) == 0
    assert B.rmsnorm_set_launch_override(4, 0, 0, 0, 0) == 0
    assert B.rmsnorm_set_launch_override(0, 33, 0, 0, 0) == 9
    assert B.rmsnorm_set_launch_override(0, 0, 9, 0, 0) == 9
    assert B.rmsnorm_set_launch_override(0, 0, -1, 0, 0) == 9
    assert B.rmsnorm_set_launch_override(0, 0, 0, 0, 0) == 0


def test_layernorm_host_validation_without_gpu():
    # layernorm_fwd(x, ldx, gamma, beta, y, ldy, mean, rstd, M, N, eps, dtype, stream)
    assert B.layernorm_fwd(None, 8, None, None, None, 8, None, None, 4, 8, 1e-5, 5, 0) == 3
    assert B.layernorm_fwd(None, 8, None, None, None, 8, None, None, 4, 0, 1e-5, 0, 0) == 2
    assert B.layernorm_fwd(None, 7, None, None, None, 8, None, None, 4, 8, 1e-5, 0, 0) == 2  # ldx < N
    assert B.layernorm_fwd(None, 8, None, None, None, 8, None, None, 4, 8, 0.0, 0, 0) == 4
    assert B.layernorm_fwd(None, 8, None, None, None, 8, None, None, 0, 8, 1e-5, 0, 0) == 0  # M == 0
    assert B.layernorm_fwd(0x1000, 8, 0x1000, None, 0x2000, 8, None, None, 4, 8, 1e-5, 0, 0) == 1
    assert B.layernorm_fwd(0x1000, 8, 0x1000, 0x1002, 0x2000, 8, None, None, 4, 8, 1e-5, 0, 0) == 5
    assert B.layernorm_fwd(0x1000, 8, 0x1000, 0x1000, 0x2000, 8, 0x3002, None, 4, 8, 1e-5, 0, 0) == 5
    # layernorm_bwd(dy, lddy, x, ldx, gamma, mean, rstd, dx, lddx, dgamma, dbeta, M, N, dtype, ws, bytes, stream)
    assert B.layernorm_bwd(None, 8, None, 8, None, None, None, None, 8, 0x1000, None, 4, 8, 0, None, 0, 0) == 1
    assert B.layernorm_bwd(None, 8, None, 8, None, None, None, None, 8, 0x1000, 0x1001, 4, 8, 1, None, 0, 0) == 5
    assert B.layernorm_bwd(None, 8, None, 8, None, None, None, None, 8, 0x1000, 0x2000, 4, 8, 0, None, 0, 0) == 1
    assert B.layernorm_bwd(0x1000, 8, 0x1000, 8, 0x1000, 0x1000, 0x1000, 0x1000, 8, 0x1000, 0x2000, 4, 8, 0,
                           0x1008, 1 << 20, 0) == 5
    assert B.layernorm_bwd(None, 8, None, 9, None, None, None, None, 8, 0x1000, 0x2000, 4, 10, 0, None, 0, 0) == 2
    assert B.layernorm_bwd_workspace_size(0, 8, 0) == 0
    assert B.layernorm_bwd_workspace_size(4, 8, 9) == 0


def test_double_backward_host_validation_without_gpu():
    # rmsnorm_bwd_bwd(ddx, ldddx, ddg, dy, lddy, x, ldx, gamma, rstd, d_dy, ldd_dy, d_x, ldd_x, d_gamma,
    #                 M, N, dtype, offset, ws, bytes, stream)
    f = B.rmsnorm_bwd_bwd
    assert f(None, 8, None, None, 8, None, 8, None, None, None, 8, None, 8, 0x1000, 4, 8, 5, 0, None, 0, 0) == 3
    assert f(None, 8, None, None, 8, None, 8, None, None, None, 8, None, 8, 0x1000, 4, 8, 0, 2, None, 0, 0) == 9
    assert f(None, 7, None, None, 8, None, 8, None, None, None, 8, None, 8, 0x1000, 4, 8, 0, 0, None, 0, 0) == 2
    assert f(None, 8, None, None, 8, None, 8, None, None, None, 8, None, 8, None, 4, 8, 0, 0, None, 0, 0) == 1
    assert f(None, 8, None, None, 8, None, 8, None, None, None, 8, None, 8, 0x1001, 4, 8, 1, 0, None, 0, 0) == 5
    assert f(None, 8, None, None, 8, None, 8, None, None, None, 8, None, 8, 0x1000, 4, 8, 0, 0, None, 0, 0) == 1
    assert B.rmsnorm_bwd_bwd_workspace_size(0, 8, 0) == 0
    assert B.rmsnorm_bwd_bwd_workspace_size(4, 8, 9) == 0


def test_library_is_in_tree_and_built_for_sm_103a():
    assert os.path.dirname(B.LIB_PATH) == os.path.dirname(os.path.abspath(B.__file__))
    assert "arch=compute_103a,code=sm_103a" in " ".join(build_mod.ARCH)
