"""Strided rows: rmsnorm_fwd_strided / rmsnorm_bwd_strided on views whose rows
are further apart than N elements.

Inputs are copied into the first N columns of wider buffers; outputs go to the
first N columns of wider buffers whose gap columns hold a sentinel that must
survive. Results are gated against the oracle on the dense rows.
"""
import numpy as np
import pytest

from oracle import check, gate
from rmsnorm_fwd_bwd_gb300 import binding as B
from rmsnorm_fwd_bwd_gb300 import inputs

pytestmark = pytest.mark.gpu

SENT = {"float32": -12345.5, "float16": 1234.0, "bfloat16": 1234.0}


@pytest.fixture(scope="module")
def torch():
    t = pytest.importorskip("torch")
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    return t


def _wide(torch, dense_np, ld, dtype):
    M, N = dense_np.shape
    t = B.to_device(dense_np.reshape(-1), dtype).view(M, N)
    buf = torch.full((M, ld), SENT[dtype], dtype=t.dtype, device="cuda")
    buf[:, :N] = t
    return buf


def _out(torch, M, N, ld, dtype):
    return torch.full((M, ld), SENT[dtype], dtype=getattr(torch, dtype), device="cuda")


# (dtype, N, ldx, lddy, ldy_and_lddx): paths -- TMA (pitches multiples of 16 B),
# row-vector (x and dy rows at equal phases), general (x and dy phases differ)
CASES = [
    ("bfloat16", 4096, 4160, 4160, 4160),
    ("bfloat16", 4096, 4100, 4100, 4100),
    ("bfloat16", 4099, 4200, 4208, 4301),
    ("float32", 8192, 8200, 8200, 8208),
    ("float16", 1000, 1003, 1003, 1024),
    ("float32", 255, 256, 257, 300),
]


@pytest.mark.parametrize("dtype,N,ldx,lddy,ldo", CASES)
@pytest.mark.parametrize("offset", [False, True])
def test_strided_rows(torch, dtype, N, ldx, lddy, ldo, offset):
    M = 67
    x, g, dy = inputs.make_inputs(M, N, dtype, seed=N + ldx, offset=offset)
    xb = _wide(torch, x, ldx, dtype)
    dyb = _wide(torch, dy, lddy, dtype)
    gt = B.to_device(g, dtype)
    yb = _out(torch, M, N, ldo, dtype)
    dxb = _out(torch, M, N, ldo, dtype)
    dg = torch.empty_like(gt)
    rstd = torch.empty(M, dtype=torch.float32, device="cuda")
    assert B.rmsnorm_fwd_strided(xb, ldx, gt, yb, ldo, rstd, M, N, 1e-6, dtype, int(offset)) == 0
    need = B.rmsnorm_bwd_workspace_size(M, N, dtype)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    assert B.rmsnorm_bwd_strided(dyb, lddy, xb, ldx, gt, rstd, dxb, ldo, dg, M, N, dtype, int(offset),
                                 ws, need) == 0
    torch.cuda.synchronize()
    for buf in (yb, dxb):
        gap = buf[:, N:]
        assert torch.all(gap == SENT[dtype]), "a gap element between rows was written"
    y = B.to_numpy(yb[:, :N].contiguous(), dtype)
    dx = B.to_numpy(dxb[:, :N].contiguous(), dtype)
    res = check.gate_outputs(x, g, dy, dtype, offset, 1e-6, y=y, rstd=B.to_numpy(rstd, "float32"),
                             dx=dx, dgamma=B.to_numpy(dg, dtype))
    assert gate.overall(res) == "PASS", gate.report(f"strided {dtype} N={N} ld={ldx},{lddy},{ldo}", res)


def test_strided_matches_dense_bitwise(torch):
    M, N, dtype = 300, 4096, "bfloat16"
    x, g, dy = inputs.make_inputs(M, N, dtype, seed=8)
    from tests import gpu_util
    dense = gpu_util.run(x, g, dy, dtype)
    xb, dyb = _wide(torch, x, 4160, dtype), _wide(torch, dy, 4160, dtype)
    gt = B.to_device(g, dtype)
    yb, dxb = _out(torch, M, N, 4160, dtype), _out(torch, M, N, 4160, dtype)
    dg = torch.empty_like(gt)
    rstd = torch.empty(M, dtype=torch.float32, device="cuda")
    assert B.rmsnorm_fwd_strided(xb, 4160, gt, yb, 4160, rstd, M, N, 1e-6, dtype, 0) == 0
    need = B.rmsnorm_bwd_workspace_size(M, N, dtype)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    assert B.rmsnorm_bwd_strided(dyb, 4160, xb, 4160, gt, rstd, dxb, 4160, dg, M, N, dtype, 0, ws, need) == 0
    torch.cuda.synchronize()
    assert np.array_equal(B.to_numpy(yb[:, :N].contiguous(), dtype), dense[0])
    assert np.array_equal(B.to_numpy(rstd, "float32"), dense[1])
    assert np.array_equal(B.to_numpy(dxb[:, :N].contiguous(), dtype), dense[2])
    assert np.array_equal(B.to_numpy(dg, dtype), dense[3])


def test_strided_rejects_short_pitch(torch):
    x = torch.zeros(4, 64, device="cuda")
    g = torch.ones(64, device="cuda")
    r = torch.empty(4, device="cuda")
    assert B.rmsnorm_fwd_strided(x, 63, g, x, 64, r, 4, 64, 1e-6, "float32", 0) == 2  # SHAPE


def test_strided_rows_with_the_row_pool(torch):
    """Rows the row pool hands out (heads and queued segments, forward and backward)
    use each tensor's own pitch: at 12000 rows the strided calls give the dense
    calls' bits and never touch the gaps between rows."""
    M, N, dtype = 12000, 4096, "bfloat16"
    for p in (0, 1):
        plan = B.rmsnorm_describe_plan(p, M, N, dtype)
        assert "pool_head=" in plan, plan
    x, g, dy = inputs.make_inputs(M, N, dtype, seed=21)
    from tests import gpu_util
    dense = gpu_util.run(x, g, dy, dtype)
    ldx, lddy, ldo = 4160, 4176, 4168
    xb, dyb = _wide(torch, x, ldx, dtype), _wide(torch, dy, lddy, dtype)
    gt = B.to_device(g, dtype)
    yb, dxb = _out(torch, M, N, ldo, dtype), _out(torch, M, N, ldo, dtype)
    dg = torch.empty_like(gt)
    rstd = torch.empty(M, dtype=torch.float32, device="cuda")
    assert B.rmsnorm_fwd_strided(xb, ldx, gt, yb, ldo, rstd, M, N, 1e-6, dtype, 0) == 0
    need = B.rmsnorm_bwd_workspace_size(M, N, dtype)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    assert B.rmsnorm_bwd_strided(dyb, lddy, xb, ldx, gt, rstd, dxb, ldo, dg, M, N, dtype, 0, ws, need) == 0
    torch.cuda.synchronize()
    for buf in (yb, dxb):
        assert torch.all(buf[:, N:] == SENT[dtype]), "a gap element between rows was written"
    assert np.array_equal(B.to_numpy(yb[:, :N].contiguous(), dtype), dense[0])
    assert np.array_equal(B.to_numpy(rstd, "float32"), dense[1])
    assert np.array_equal(B.to_numpy(dxb[:, :N].contiguous(), dtype), dense[2])
    assert np.array_equal(B.to_numpy(dg, dtype), dense[3])
