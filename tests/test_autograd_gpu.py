"""PyTorch integration on the GPU: autograd through the C-ABI kernels.

Follows the integration evidence of the page "Check an AI model calculation
before accelerating it" (section "Connecting Autograd and actually training"):
gradients through the adapter, call counters proving the kernel path ran, a tiny
Linear -> RMSNorm -> SiLU -> Linear network trained for 100 Adam steps on
synthetic data next to a plain-PyTorch RMSNorm from the same initialisation,
and a save/reload of the weights. And, as on the torchtitan numerics page's
contract tests, torch.library.opcheck and a trace without graph breaks.
"""
import numpy as np
import pytest

from oracle import check, gate
from rmsnorm_fwd_bwd_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = pytest.importorskip("torch")
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    return t


@pytest.fixture(scope="module")
def ag(torch):
    from rmsnorm_fwd_bwd_gb300 import autograd
    return autograd


@pytest.mark.parametrize("dtype,offset", [("bfloat16", False), ("float16", True), ("float32", False)])
def test_autograd_gradients_pass_the_gate(torch, ag, dtype, offset):
    from rmsnorm_fwd_bwd_gb300 import binding as B
    M, N = 96, 1536
    x, g, dy = inputs.make_inputs(M, N, dtype, seed=17, offset=offset)
    xt = B.to_device(x.reshape(-1), dtype).view(4, 24, N).requires_grad_(True)
    gt = B.to_device(g, dtype).requires_grad_(True)
    dyt = B.to_device(dy.reshape(-1), dtype).view(4, 24, N)
    y = ag.rms_norm(xt, gt, 1e-6, offset)
    y.backward(dyt)
    res = check.gate_outputs(x, g, dy, dtype, offset, 1e-6,
                             y=B.to_numpy(y, dtype).reshape(M, N),
                             dx=B.to_numpy(xt.grad, dtype).reshape(M, N),
                             dgamma=B.to_numpy(gt.grad, dtype))
    assert gate.overall(res) == "PASS", gate.report(f"autograd {dtype}", res)


def _torch_rmsnorm(torch, x, w, eps):
    r = torch.rsqrt(x.float().square().mean(-1, keepdim=True) + eps)
    return (x.float() * r * w.float()).to(x.dtype)


def test_tiny_training_run_and_reload(torch, ag, tmp_path):
    torch.manual_seed(0)
    D, H = 64, 96

    def make(norm):
        return torch.nn.Sequential(torch.nn.Linear(D, H), norm, torch.nn.SiLU(),
                                   torch.nn.Linear(H, 1)).cuda()

    class TorchNorm(torch.nn.Module):
        def __init__(self):
            super().__init__()
            self.weight = torch.nn.Parameter(torch.ones(H, device="cuda"))

        def forward(self, x):
            return _torch_rmsnorm(torch, x, self.weight, 1e-6)

    ours = make(ag.RMSNorm(H, device="cuda"))
    ref = make(TorchNorm())
    ref.load_state_dict(ours.state_dict())          # identical initialisation
    gen = torch.Generator().manual_seed(1)
    w_true = torch.randn(D, 1, generator=gen)
    xs = torch.randn(3200 + 640, D, generator=gen)
    ys = torch.tanh(xs @ w_true) + 0.1 * torch.randn(xs.shape[0], 1, generator=gen)
    train_x, train_y = xs[:3200].cuda(), ys[:3200].cuda()
    test_x, test_y = xs[3200:].cuda(), ys[3200:].cuda()

    with torch.no_grad():
        e_out = (ours(test_x) - ref(test_x)).abs().max().item()
    assert e_out < 1e-5

    before = dict(ag.CALLS)
    opt_a = torch.optim.Adam(ours.parameters(), lr=1e-3)
    opt_b = torch.optim.Adam(ref.parameters(), lr=1e-3)
    for step in range(100):
        bx, by = train_x[step * 32:(step + 1) * 32], train_y[step * 32:(step + 1) * 32]
        for model, opt in ((ours, opt_a), (ref, opt_b)):
            opt.zero_grad(set_to_none=True)
            loss = torch.nn.functional.mse_loss(model(bx), by)
            loss.backward()
            opt.step()
    assert ag.CALLS["forward"] - before["forward"] == 100
    assert ag.CALLS["backward"] - before["backward"] == 100
    with torch.no_grad():
        mse_a = torch.nn.functional.mse_loss(ours(test_x), test_y).item()
        mse_b = torch.nn.functional.mse_loss(ref(test_x), test_y).item()
    assert abs(mse_a - mse_b) <= 1e-3 * max(mse_b, 1e-6)
    # weights-only save and reload reproduce the outputs exactly
    path = tmp_path / "tiny.pt"
    torch.save(ours.state_dict(), path)
    again = make(ag.RMSNorm(H, device="cuda"))
    again.load_state_dict(torch.load(path))
    with torch.no_grad():
        assert torch.equal(again(test_x), ours(test_x))


def test_opcheck_and_trace_without_graph_breaks(torch, ag):
    x = torch.randn(8, 6, 256, device="cuda", dtype=torch.bfloat16, requires_grad=True)
    w = (1 + 0.1 * torch.randn(256, device="cuda")).to(torch.bfloat16).requires_grad_(True)
    torch.library.opcheck(torch.ops.rmsnorm_gb300.fwd.default, (x, w, 1e-6, False))
    compiled = torch.compile(lambda a, b: ag.rms_norm(a, b, 1e-6, False), fullgraph=True, backend="eager")
    y1 = compiled(x, w)
    y2 = ag.rms_norm(x, w, 1e-6, False)
    assert torch.equal(y1, y2)
    g = torch.randn_like(y1)
    (gx1, gw1) = torch.autograd.grad(y1, (x, w), g)
    (gx2, gw2) = torch.autograd.grad(y2, (x, w), g)
    assert torch.equal(gx1, gx2) and torch.equal(gw1, gw2)


def test_strided_view_passes_the_gate(torch, ag):
    """A 2-D view of the first N columns of a wider tensor goes to the kernels
    with its row pitch. (Its rows are not 16-byte multiples apart, so it takes
    another kernel path than a contiguous copy would: the results agree within
    the gate, not bit for bit.)"""
    from rmsnorm_fwd_bwd_gb300 import binding as B
    M, N, ld, dtype = 64, 1000, 1100, "bfloat16"
    x, g, dy = inputs.make_inputs(M, N, dtype, seed=23)
    big = torch.zeros(M, ld, device="cuda", dtype=torch.bfloat16)
    big[:, :N] = B.to_device(x.reshape(-1), dtype).view(M, N)
    xv = big[:, :N].detach().requires_grad_(True)
    assert xv.stride() == (ld, 1)
    w = B.to_device(g, dtype).requires_grad_(True)
    y = ag.rms_norm(xv, w)
    y.backward(B.to_device(dy.reshape(-1), dtype).view(M, N))
    res = check.gate_outputs(x, g, dy, dtype, False, 1e-6,
                             y=B.to_numpy(y, dtype).reshape(M, N),
                             dx=B.to_numpy(xv.grad, dtype).reshape(M, N),
                             dgamma=B.to_numpy(w.grad, dtype))
    assert gate.overall(res) == "PASS", gate.report("autograd strided view", res)


def test_module_rejects_mismatched_weight(torch, ag):
    x = torch.randn(4, 32, device="cuda")
    with pytest.raises(ValueError):
        ag.rms_norm(x, torch.ones(31, device="cuda"))
    with pytest.raises(ValueError):
        ag.rms_norm(x, torch.ones(32, device="cuda", dtype=torch.float16))


# --------------------------------------------------------------------------- #
# LayerNorm through the same adapter pattern
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("dtype", ["bfloat16", "float16", "float32"])
def test_layer_norm_gradients_pass_the_gate(torch, ag, dtype):
    from rmsnorm_fwd_bwd_gb300 import binding as B
    M, N = 96, 1536
    x, g, b, dy = inputs.make_ln_inputs(M, N, dtype, seed=19)
    xt = B.to_device(x.reshape(-1), dtype).view(4, 24, N).requires_grad_(True)
    gt = B.to_device(g, dtype).requires_grad_(True)
    bt = B.to_device(b, dtype).requires_grad_(True)
    dyt = B.to_device(dy.reshape(-1), dtype).view(4, 24, N)
    y = ag.layer_norm(xt, gt, bt, 1e-5)
    y.backward(dyt)
    res = check.gate_ln_outputs(x, g, b, dy, dtype, 1e-5,
                                y=B.to_numpy(y, dtype).reshape(M, N),
                                dx=B.to_numpy(xt.grad, dtype).reshape(M, N),
                                dgamma=B.to_numpy(gt.grad, dtype), dbeta=B.to_numpy(bt.grad, dtype))
    assert gate.overall(res) == "PASS", gate.report(f"layer_norm autograd {dtype}", res)


def test_layer_norm_training_run_matches_torch(torch, ag):
    torch.manual_seed(0)
    D, H = 64, 96

    def make(norm):
        return torch.nn.Sequential(torch.nn.Linear(D, H), norm, torch.nn.SiLU(),
                                   torch.nn.Linear(H, 1)).cuda()

    ours = make(ag.LayerNorm(H, device="cuda"))
    ref = make(torch.nn.LayerNorm(H, eps=1e-5, device="cuda"))
    ref.load_state_dict(ours.state_dict())          # identical initialisation
    gen = torch.Generator().manual_seed(2)
    w_true = torch.randn(D, 1, generator=gen)
    xs = torch.randn(3200 + 640, D, generator=gen)
    ys = torch.tanh(xs @ w_true) + 0.1 * torch.randn(xs.shape[0], 1, generator=gen)
    train_x, train_y = xs[:3200].cuda(), ys[:3200].cuda()
    test_x, test_y = xs[3200:].cuda(), ys[3200:].cuda()
    with torch.no_grad():
        assert (ours(test_x) - ref(test_x)).abs().max().item() < 1e-5
    before = dict(ag.LN_CALLS)
    opt_a = torch.optim.Adam(ours.parameters(), lr=1e-3)
    opt_b = torch.optim.Adam(ref.parameters(), lr=1e-3)
    for step in range(100):
        bx, by = train_x[step * 32:(step + 1) * 32], train_y[step * 32:(step + 1) * 32]
        for model, opt in ((ours, opt_a), (ref, opt_b)):
            opt.zero_grad(set_to_none=True)
            torch.nn.functional.mse_loss(model(bx), by).backward()
            opt.step()
    assert ag.LN_CALLS["forward"] - before["forward"] == 100
    assert ag.LN_CALLS["backward"] - before["backward"] == 100
    with torch.no_grad():
        mse_a = torch.nn.functional.mse_loss(ours(test_x), test_y).item()
        mse_b = torch.nn.functional.mse_loss(ref(test_x), test_y).item()
    assert abs(mse_a - mse_b) <= 1e-3 * max(mse_b, 1e-6)


def test_layer_norm_opcheck_and_trace(torch, ag):
    x = torch.randn(8, 6, 256, device="cuda", dtype=torch.bfloat16, requires_grad=True)
    w = (1 + 0.1 * torch.randn(256, device="cuda")).to(torch.bfloat16).requires_grad_(True)
    b = (0.1 * torch.randn(256, device="cuda")).to(torch.bfloat16).requires_grad_(True)
    torch.library.opcheck(torch.ops.rmsnorm_gb300.ln_fwd.default, (x, w, b, 1e-5))
    compiled = torch.compile(lambda a, c, d: ag.layer_norm(a, c, d, 1e-5), fullgraph=True, backend="eager")
    y1 = compiled(x, w, b)
    y2 = ag.layer_norm(x, w, b, 1e-5)
    assert torch.equal(y1, y2)
    g = torch.randn_like(y1)
    g1 = torch.autograd.grad(y1, (x, w, b), g)
    g2 = torch.autograd.grad(y2, (x, w, b), g)
    assert all(torch.equal(p, q) for p, q in zip(g1, g2))


def test_layer_norm_strided_view(torch, ag):
    from rmsnorm_fwd_bwd_gb300 import binding as B
    M, N, ld, dtype = 64, 1000, 1100, "bfloat16"
    x, g, b, dy = inputs.make_ln_inputs(M, N, dtype, seed=29)
    big = torch.zeros(M, ld, device="cuda", dtype=torch.bfloat16)
    big[:, :N] = B.to_device(x.reshape(-1), dtype).view(M, N)
    xv = big[:, :N].detach().requires_grad_(True)
    w = B.to_device(g, dtype).requires_grad_(True)
    bb = B.to_device(b, dtype).requires_grad_(True)
    y = ag.layer_norm(xv, w, bb)
    y.backward(B.to_device(dy.reshape(-1), dtype).view(M, N))
    res = check.gate_ln_outputs(x, g, b, dy, dtype, 1e-5,
                                y=B.to_numpy(y, dtype).reshape(M, N),
                                dx=B.to_numpy(xv.grad, dtype).reshape(M, N),
                                dgamma=B.to_numpy(w.grad, dtype), dbeta=B.to_numpy(bb.grad, dtype))
    assert gate.overall(res) == "PASS", gate.report("layer_norm strided view", res)
