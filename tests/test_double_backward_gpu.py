"""GPU parity of the RMSNorm double backward (rmsnorm_bwd_bwd) against the CPU
oracle, and second-order autograd through rms_norm.

Every case gates d_dy, d_x and d_gamma with the golden / reference / target
gate. Shapes cover the narrow-row path (rows of at most 2 KB), the TMA path,
the cluster path (rows over 4096 elements), the ragged TMA path (rows off 16
bytes: odd row lengths, shifted pointers, odd pitches, outputs at another
phase), the general path (inputs at different phases, rows too wide for the
ragged ring), the offset variant, an absent ddgamma, empty inputs, strided rows
and the headline shape at full size on sampled rows.
"""
import numpy as np
import pytest

from oracle import check, gate
from rmsnorm_fwd_bwd_gb300 import inputs

from . import gpu_util

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rmsnorm_fwd_bwd_gb300 import binding
    binding.rmsnorm_device_error(clear=True)
    yield
    assert binding.rmsnorm_device_error(clear=True) == 0, "a kernel reported a wait timeout"


def _cotangents(M, N, dtype, seed, with_ddg=True):
    ddx = inputs.to_storage(inputs.normal(seed, 3, (M, N)), dtype)
    ddg = inputs.to_storage(inputs.normal(seed, 4, (N,)), dtype) if with_ddg else None
    return ddx, ddg


def _gate(M, N, dtype, seed, offset=False, with_ddg=True, misalign=False, title=""):
    x, g, dy = inputs.make_inputs(M, N, dtype, seed=seed, offset=offset)
    ddx, ddg = _cotangents(M, N, dtype, seed, with_ddg)
    d_dy, d_x, d_g = gpu_util.dbwd_run(ddx, ddg, dy, x, g, dtype, offset=offset, misalign=misalign)
    res = check.gate_bwd_bwd_outputs(ddx, ddg, dy, x, g, dtype, offset, 1e-6, d_dy=d_dy, d_x=d_x, d_gamma=d_g)
    text = gate.report(title or f"double backward {dtype} {M}x{N} offset={offset}", res)
    print("\n" + text)
    assert gate.overall(res) == "PASS", text
    return d_dy, d_x, d_g


def _plan(M, N, dtype, aligned16=1):
    from rmsnorm_fwd_bwd_gb300 import binding as B
    return B.rmsnorm_describe_plan(4, M, N, dtype, aligned16)


SHAPES = [
    # narrow rows (at most 2 KB): a row per group of lanes, every (lanes, vectors) instance
    ("bfloat16", 77, 8, "lanes lanes=4 kv=1 "),
    ("bfloat16", 65, 64, "lanes lanes=4 kv=2 "),
    ("bfloat16", 300, 128, "lanes lanes=8 kv=2 "),
    ("float32", 64, 256, "lanes lanes=32 kv=2 "),
    ("bfloat16", 99, 256, "lanes lanes=16 kv=2 "),
    ("bfloat16", 130, 768, "lanes lanes=32 kv=3 "),
    ("float16", 129, 1000, "lanes lanes=32 kv=4 "),
    ("bfloat16", 300, 2048, "tma cluster=1"),
    ("bfloat16", 300, 4096, "tma cluster=1"),
    ("float32", 41, 8192, "tma cluster=2"),
    ("bfloat16", 40, 16384, "tma cluster=8"),
    ("float32", 24, 16384, "tma cluster=8"),
    ("bfloat16", 67, 4099, "ragged"),
    ("float32", 50, 333, "ragged"),
    ("float16", 33, 1001, "ragged"),
    ("bfloat16", 9, 3, "ragged"),
    ("float32", 19, 4099, "ragged"),
    ("bfloat16", 20, 7001, "ragged"),
    ("bfloat16", 20, 8001, "scalar"),
    ("float32", 16, 5001, "scalar"),
    # the ragged ring's limits: 320 threads x 3 vectors (2-byte), a 16 KB + 32 byte span (fp32)
    ("bfloat16", 9, 7671, "ragged"),
    ("bfloat16", 9, 7673, "scalar"),
    ("float32", 9, 4101, "scalar"),
]


@pytest.mark.parametrize("dtype,M,N,path", SHAPES)
@pytest.mark.parametrize("offset", [False, True])
def test_shapes_and_paths(dtype, M, N, path, offset):
    assert _plan(M, N, dtype).startswith(path)
    _gate(M, N, dtype, seed=N + M, offset=offset)


@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
@pytest.mark.parametrize("N", [256, 2048])
def test_without_ddgamma(dtype, N):
    _gate(96, N, dtype, seed=5, with_ddg=False, title=f"double backward {dtype} N={N} ddgamma absent")


@pytest.mark.parametrize("dtype", ["float32", "float16", "bfloat16"])
@pytest.mark.parametrize("offset", [False, True])
def test_shifted_pointers_take_the_ragged_path(dtype, offset):
    # every tensor one element off a 16-byte boundary: x, dy and ddx share a phase
    assert _plan(45, 2048, dtype, aligned16=0).startswith("ragged")
    _gate(45, 2048, dtype, seed=11, offset=offset, misalign=True, title=f"double backward {dtype} shifted")


@pytest.mark.parametrize("names", [{"x"}, {"dy"}, {"ddx"}, {"d_dy"}, {"d_x"}, {"ddx", "dy", "x"}])
@pytest.mark.parametrize("N", [2048, 4099])
def test_partly_shifted_pointers(names, N):
    # inputs at different phases take the general path; outputs at any phase get
    # element stores on the ragged path
    _gate(37, N, "bfloat16", seed=12, misalign=names, title=f"double backward shifted {sorted(names)} N={N}")


def test_repeated_runs_are_bitwise_identical():
    x, g, dy = inputs.make_inputs(700, 4096, "bfloat16", seed=13)
    ddx, ddg = _cotangents(700, 4096, "bfloat16", 13)
    first = gpu_util.dbwd_run(ddx, ddg, dy, x, g, "bfloat16")
    again = gpu_util.dbwd_run(ddx, ddg, dy, x, g, "bfloat16")
    for a, b in zip(first, again):
        assert np.array_equal(a, b)


def test_empty_rows_zero_d_gamma():
    import torch
    from rmsnorm_fwd_bwd_gb300 import binding as B
    N = 300
    dg = torch.full((N,), 7.0, device="cuda")
    e = torch.empty(0, device="cuda")
    g = torch.ones(N, device="cuda")
    assert B.rmsnorm_bwd_bwd_workspace_size(0, N, "float32") == 0
    assert B.rmsnorm_bwd_bwd(e, N, None, e, N, e, N, g, e, e, N, e, N, dg, 0, N, "float32", 0, None, 0) == 0
    torch.cuda.synchronize()
    assert torch.all(dg == 0)


@pytest.mark.parametrize("M,N,ld,ld_out", [(67, 4096, 4160, 4160), (67, 4099, 4111, 4100), (29, 1001, 1001, 1013)])
def test_strided_rows(M, N, ld, ld_out):
    # pitches (elements) of the inputs and of the outputs; odd pitches put the rows
    # of one tensor at eight different 16-byte phases
    import torch
    from rmsnorm_fwd_bwd_gb300 import binding as B
    dtype = "bfloat16"
    x, g, dy = inputs.make_inputs(M, N, dtype, seed=21)
    ddx, ddg = _cotangents(M, N, dtype, 21)

    def wide(a, pitch):
        buf = torch.full((M, pitch), 1234.0, dtype=torch.bfloat16, device="cuda")
        if a is not None:
            buf[:, :N] = B.to_device(a.reshape(-1), dtype).view(M, N)
        return buf

    xb, dyb, tb = wide(x, ld), wide(dy, ld), wide(ddx, ld)
    gt, qt = B.to_device(g, dtype), B.to_device(ddg, dtype)
    rstd = torch.empty(M, device="cuda")
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    assert B.rmsnorm_fwd_strided(xb, ld, gt, y, N, rstd, M, N, 1e-6, dtype, 0) == 0
    o_dy, o_x = wide(None, ld_out), wide(None, ld_out)
    o_g = torch.empty_like(gt)
    need = B.rmsnorm_bwd_bwd_workspace_size(M, N, dtype)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    assert B.rmsnorm_bwd_bwd(tb, ld, qt, dyb, ld, xb, ld, gt, rstd, o_dy, ld_out, o_x, ld_out, o_g, M, N, dtype, 0,
                             ws, need) == 0
    torch.cuda.synchronize()
    assert torch.all(o_dy[:, N:] == 1234.0) and torch.all(o_x[:, N:] == 1234.0)
    res = check.gate_bwd_bwd_outputs(ddx, ddg, dy, x, g, dtype, False, 1e-6,
                                     d_dy=B.to_numpy(o_dy[:, :N].contiguous(), dtype),
                                     d_x=B.to_numpy(o_x[:, :N].contiguous(), dtype), d_gamma=B.to_numpy(o_g, dtype))
    assert gate.overall(res) == "PASS", gate.report(f"double backward strided {M}x{N} ld={ld}/{ld_out}", res)


def test_ragged_sampled_rows_at_65536():
    """bf16 65536x4099 on the ragged ring: d_dy and d_x gated on sampled rows,
    d_gamma in full."""
    M, N, dtype = 65536, 4099, "bfloat16"
    assert _plan(M, N, dtype, aligned16=0).startswith("ragged")
    x, g, dy = inputs.make_inputs(M, N, dtype, seed=31)
    ddx, ddg = _cotangents(M, N, dtype, 31)
    d_dy, d_x, d_g = gpu_util.dbwd_run(ddx, ddg, dy, x, g, dtype)
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([np.arange(24), np.arange(M - 24, M), rng.choice(M, 120, replace=False)]))
    res = check.gate_bwd_bwd_outputs(ddx, ddg, dy, x, g, dtype, False, 1e-6, d_dy=d_dy[rows], d_x=d_x[rows],
                                     rows=rows)
    res += check.gate_bwd_bwd_outputs(ddx, ddg, dy, x, g, dtype, False, 1e-6, d_gamma=d_g)
    assert gate.overall(res) == "PASS", gate.report("double backward bf16 65536x4099", res)


def test_headline_shape_sampled_rows():
    """bf16 65536x4096, the headline shape: d_dy and d_x gated on sampled rows,
    d_gamma in full."""
    w = inputs.WORKLOADS["bf16_65536x4096"]
    x, g, dy = inputs.workload_inputs(w)
    ddx, ddg = _cotangents(w.M, w.N, w.dtype, 77)
    d_dy, d_x, d_g = gpu_util.dbwd_run(ddx, ddg, dy, x, g, w.dtype)
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([np.arange(32), np.arange(w.M - 32, w.M), rng.choice(w.M, 160, replace=False)]))
    res = check.gate_bwd_bwd_outputs(ddx, ddg, dy, x, g, w.dtype, False, w.eps, d_dy=d_dy[rows], d_x=d_x[rows],
                                     rows=rows)
    res += check.gate_bwd_bwd_outputs(ddx, ddg, dy, x, g, w.dtype, False, w.eps, d_gamma=d_g)
    assert gate.overall(res) == "PASS", gate.report("double backward bf16 65536x4096", res)


# --------------------------------------------------------------------------- #
# second-order autograd through rms_norm
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("dtype,offset", [("float32", False), ("bfloat16", True)])
def test_autograd_second_order(dtype, offset):
    import torch
    from rmsnorm_fwd_bwd_gb300 import autograd as ag
    from rmsnorm_fwd_bwd_gb300 import binding as B
    M, N = 64, 1024
    x, g, dy = inputs.make_inputs(M, N, dtype, seed=31, offset=offset)
    ddx, ddg = _cotangents(M, N, dtype, 31)
    xt = B.to_device(x.reshape(-1), dtype).view(M, N).requires_grad_(True)
    gt = B.to_device(g, dtype).requires_grad_(True)
    dyt = B.to_device(dy.reshape(-1), dtype).view(M, N).requires_grad_(True)
    before = ag.CALLS["double_backward"]
    y = ag.rms_norm(xt, gt, 1e-6, offset)
    dx, dg = torch.autograd.grad(y, (xt, gt), dyt, create_graph=True)
    ddxt = B.to_device(ddx.reshape(-1), dtype).view(M, N)
    ddgt = B.to_device(ddg, dtype)
    d_dy, d_x, d_g = torch.autograd.grad((dx, dg), (dyt, xt, gt), (ddxt, ddgt))
    assert ag.CALLS["double_backward"] == before + 1
    res = check.gate_bwd_bwd_outputs(ddx, ddg, dy, x, g, dtype, offset, 1e-6,
                                     d_dy=B.to_numpy(d_dy, dtype), d_x=B.to_numpy(d_x, dtype),
                                     d_gamma=B.to_numpy(d_g, dtype))
    assert gate.overall(res) == "PASS", gate.report(f"autograd second order {dtype}", res)


def test_autograd_gradient_penalty_matches_torch_composite():
    """A gradient penalty (the norm of dL/dx) trained through rms_norm agrees
    with the same penalty through a plain-PyTorch fp32 RMSNorm."""
    import torch
    from rmsnorm_fwd_bwd_gb300 import autograd as ag
    torch.manual_seed(0)
    x = torch.randn(32, 512, device="cuda", requires_grad=True)
    w = (1 + 0.1 * torch.randn(512, device="cuda")).requires_grad_(True)
    t = torch.randn(32, 512, device="cuda")

    def penalty(norm):
        y = norm(x, w)
        loss = ((y - t) ** 2).mean()
        gx, = torch.autograd.grad(loss, x, create_graph=True)
        return (gx ** 2).sum()

    def torch_norm(a, b):
        return a * torch.rsqrt(a.square().mean(-1, keepdim=True) + 1e-6) * b

    p1 = penalty(lambda a, b: ag.rms_norm(a, b, 1e-6))
    gx1, gw1 = torch.autograd.grad(p1, (x, w))
    p2 = penalty(torch_norm)
    gx2, gw2 = torch.autograd.grad(p2, (x, w))
    assert abs(p1.item() - p2.item()) <= 1e-5 * abs(p2.item())
    assert (gx1 - gx2).abs().max().item() <= 1e-4 * gx2.abs().max().item()
    assert (gw1 - gw2).abs().max().item() <= 1e-4 * gw2.abs().max().item()
