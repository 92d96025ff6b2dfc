"""rmsnorm_bwd_static_scratch: the backward for callers that cannot allocate.

Some callers cannot call cudaMalloc (for example a plugin whose host framework
owns all device memory). This entry point keeps the backward's partial sums in
a fixed array inside the library instead of a caller workspace. The test calls
it through the C ABI twice in a row -- two different shapes, and the second
call overwriting what the first left in the shared array -- and checks each
result against the workspace entry point rmsnorm_bwd and against the CPU
oracle's correctness gate used by the other GPU tests.

This file is named to be collected last, so that a run stopping at its first
failure has already run every other test.
"""
import numpy as np
import pytest

from oracle import check, gate
from rmsnorm_fwd_bwd_gb300 import binding as B
from rmsnorm_fwd_bwd_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = pytest.importorskip("torch")
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    return t


def _backward_both_ways(torch, x_np, g_np, dy_np, dtype, offset):
    M, N = x_np.shape
    x = B.to_device(x_np.reshape(-1), dtype)
    g = B.to_device(g_np, dtype)
    dy = B.to_device(dy_np.reshape(-1), dtype)
    y = torch.empty_like(x)
    rstd = torch.empty(M, dtype=torch.float32, device="cuda")
    assert B.rmsnorm_fwd(x, g, y, rstd, M, N, 1e-6, dtype, int(offset)) == B.RMSNORM_OK
    # existing entry point, caller workspace
    need = B.rmsnorm_bwd_workspace_size(M, N, dtype)
    assert 0 < need <= (16 << 20)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    dx_ws, dg_ws = torch.empty_like(x), torch.empty_like(g)
    assert B.rmsnorm_bwd(dy, x, g, rstd, dx_ws, dg_ws, M, N, dtype, int(offset), ws,
                         need) == B.RMSNORM_OK
    # the entry point that allocates nothing
    dx_st, dg_st = torch.full_like(x, 7), torch.full_like(g, 7)
    assert B.rmsnorm_bwd_static_scratch(dy, x, g, rstd, dx_st, dg_st, M, N, dtype,
                                        int(offset)) == B.RMSNORM_OK
    torch.cuda.synchronize()
    return (B.to_numpy(rstd, "float32"),
            B.to_numpy(dx_ws, dtype).reshape(M, N), B.to_numpy(dg_ws, dtype),
            B.to_numpy(dx_st, dtype).reshape(M, N), B.to_numpy(dg_st, dtype))


@pytest.mark.parametrize("second", [("float32", 515, 16384, True), ("bfloat16", 2048, 4096, False)])
def test_static_scratch_backward_matches_workspace_backward(torch, second):
    calls = [("bfloat16", 4096, 4096, False), second]
    for dtype, M, N, offset in calls:
        x, g, dy = inputs.make_inputs(M, N, dtype, seed=M + N, offset=offset)
        rstd, dx_ws, dg_ws, dx_st, dg_st = _backward_both_ways(torch, x, g, dy, dtype, offset)
        # same launch plan and kernels as rmsnorm_bwd: identical results
        assert np.array_equal(dx_st, dx_ws)
        assert np.array_equal(dg_st, dg_ws)
        # and within the gate every other GPU test applies
        res = check.gate_outputs(x, g, dy, dtype, offset, 1e-6, dx=dx_st, dgamma=dg_st)
        text = gate.report(f"static scratch {dtype} {M}x{N} offset={offset}", res)
        print("\n" + text)
        assert gate.overall(res) == "PASS", text
    assert B.rmsnorm_device_error(clear=True) == 0


def test_static_scratch_rejects_bad_arguments_without_launching(torch):
    N = 256
    g = torch.ones(N, device="cuda")
    dg = torch.full((N,), 5.0, device="cuda")
    assert B.rmsnorm_bwd_static_scratch(None, None, g, None, None, dg, 4, N, "float32", 0) == 1
    assert B.rmsnorm_bwd_static_scratch(None, None, g, None, None, dg, 4, 16385, "float32", 0) == 2
    torch.cuda.synchronize()
    assert torch.all(dg == 5.0)


def test_static_scratch_call_allocates_nothing(torch):
    """The defining property: a call takes no device memory. A warm-up call of
    another shape loads the library's array (with lazy module loading, the
    first use of the array's module places it on the device), and the shape's
    kernels are loaded through rmsnorm_bwd (a kernel's first launch may load its
    code); then the device's free memory is read around the first static-scratch
    calls of the shape and must not move. (Shapes too large for the array are
    rejected by the same workspace check rmsnorm_bwd applies, exercised with a
    short workspace in test_parity_gpu.py: on a 152-SM GB300 every legal shape
    fits in the 16 MiB.)"""
    wx, wg, wdy = inputs.make_inputs(64, 1024, "bfloat16", seed=3)
    _backward_both_ways(torch, wx, wg, wdy, "bfloat16", False)
    dtype, M, N, offset = "float32", 300, 8192, True
    x_np, g_np, dy_np = inputs.make_inputs(M, N, dtype, seed=11, offset=offset)
    x, g, dy = (B.to_device(a.reshape(-1), dtype) for a in (x_np, g_np, dy_np))
    y, dx = torch.empty_like(x), torch.empty_like(x)
    rstd = torch.empty(M, dtype=torch.float32, device="cuda")
    dg = torch.empty_like(g)
    need = B.rmsnorm_bwd_workspace_size(M, N, dtype)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    assert B.rmsnorm_fwd(x, g, y, rstd, M, N, 1e-6, dtype, int(offset)) == B.RMSNORM_OK
    assert B.rmsnorm_bwd(dy, x, g, rstd, dx, dg, M, N, dtype, int(offset), ws, need) == B.RMSNORM_OK
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    torch_before = torch.cuda.memory_allocated()
    for _ in range(2):
        assert B.rmsnorm_bwd_static_scratch(dy, x, g, rstd, dx, dg, M, N, dtype, int(offset)) == B.RMSNORM_OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    assert torch.cuda.memory_allocated() == torch_before
    assert B.rmsnorm_device_error(clear=True) == 0
