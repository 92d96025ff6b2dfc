"""GPU: the RMSNorm backward's row pool (per-CTA heads, then a queue of row
segments with a partial row each) against the oracle, against the static
assignment, and with every kind of leftover in the workspace's queue word."""
import numpy as np
import pytest

from oracle import check, gate
from rmsnorm_fwd_bwd_gb300 import inputs

from . import gpu_util

pytestmark = pytest.mark.gpu

# (M, N, dtype, offset): one-CTA TMA plans with at least 4 rows per CTA whose pool
# kernel (one producer warp more per CTA) keeps the plan's residency; 1, 2 and 4
# vectors per thread, 96-256 consumer threads, 2 and 3 stages
CASES = [(10000, 4096, "bfloat16", False), (10001, 4096, "bfloat16", True), (1000, 8192, "float16", True),
         (10000, 2048, "float32", True), (12000, 1024, "float32", False), (12000, 2048, "bfloat16", False),
         (12000, 3072, "float16", True), (20000, 512, "float32", False)]
BASE = (10000, 4096, "bfloat16")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rmsnorm_fwd_bwd_gb300 import binding
    binding.rmsnorm_device_error(clear=True)
    yield
    binding.rmsnorm_set_row_pool(True)
    assert binding.rmsnorm_device_error(clear=True) == 0, "a kernel reported a wait timeout"


def _gate(x, g, dy, dtype, offset, outs, title):
    y, r, dx, dg = outs
    res = check.gate_outputs(x, g, dy, dtype, offset, 1e-6, y=y, rstd=r, dx=dx, dgamma=dg)
    text = gate.report(title, res)
    print("\n" + text)
    assert gate.overall(res) == "PASS", text


def _plan(M, N, dtype):
    from rmsnorm_fwd_bwd_gb300 import binding as B
    return B.rmsnorm_describe_plan(1, M, N, dtype)


def test_pool_plans():
    """The headline shape and the base case take the pool; plans whose pool kernel
    would lose residency (four 128-thread CTAs per SM at few rows) do not."""
    assert "pool_head=" in _plan(65536, 4096, "bfloat16")
    assert "pool_head=" in _plan(*BASE)
    for M, N, dtype, _ in CASES:
        print(M, N, dtype, _plan(M, N, dtype))


@pytest.mark.parametrize("M,N,dtype,offset", CASES)
def test_pool_backward_gated(M, N, dtype, offset):
    plan = _plan(M, N, dtype)
    if "pool_head=" not in plan:
        pytest.skip(f"no row pool in this plan: {plan}")
    x, g, dy = inputs.make_inputs(M, N, dtype, seed=M + N, offset=offset)
    _gate(x, g, dy, dtype, offset, gpu_util.run(x, g, dy, dtype, offset=offset), f"pool {plan}")


@pytest.mark.parametrize("M,N,dtype,offset", CASES[:4])
def test_pool_against_static_assignment(M, N, dtype, offset):
    if "pool_head=" not in _plan(M, N, dtype):
        pytest.skip("no row pool in this plan")
    """dx does not depend on which CTA ran a row: bitwise equal. dgamma sums the
    rows in another grouping: both gated against the oracle."""
    from rmsnorm_fwd_bwd_gb300 import binding as B
    x, g, dy = inputs.make_inputs(M, N, dtype, seed=7 * M + N, offset=offset)
    pooled = gpu_util.run(x, g, dy, dtype, offset=offset)
    assert B.rmsnorm_set_row_pool(False) == 0
    try:
        plan = _plan(M, N, dtype)
        assert "pool_head=" not in plan, plan
        static = gpu_util.run(x, g, dy, dtype, offset=offset)
    finally:
        assert B.rmsnorm_set_row_pool(True) == 0
    assert np.array_equal(pooled[2], static[2])
    _gate(x, g, dy, dtype, offset, pooled, "pool")
    _gate(x, g, dy, dtype, offset, static, "static")


@pytest.mark.parametrize("fill", [0x00, 0xFF, 0x7F, "random"])
def test_pool_ignores_leftover_queue_words(fill):
    """The queue word is {ticket, next segment}: zeros, all ones (the counter's
    carry into the ticket), a large count, random bytes and the previous call's
    word all start a fresh queue: the same bits as a first call."""
    M, N, dtype = BASE
    x, g, dy = inputs.make_inputs(M, N, dtype, seed=11)
    ref = gpu_util.run(x, g, dy, dtype, ws_fill=0)
    got = gpu_util.run(x, g, dy, dtype, ws_fill=fill)
    for a, b in zip(ref, got):
        assert np.array_equal(a, b)


def test_pool_reuses_one_workspace():
    """Back-to-back calls on one workspace (each finds the previous call's ticket)
    and on one stream give identical bits."""
    torch = pytest.importorskip("torch")
    from rmsnorm_fwd_bwd_gb300 import binding as B
    M, N, dtype = BASE
    x, g, dy = inputs.make_inputs(M, N, dtype, seed=12)
    xt, gt, dyt = (B.to_device(a.reshape(-1), dtype) for a in (x, g, dy))
    y = torch.empty_like(xt)
    r = torch.empty(M, dtype=torch.float32, device="cuda")
    assert B.rmsnorm_fwd(xt, gt, y, r, M, N, 1e-6, dtype, 0) == 0
    wsz = B.rmsnorm_bwd_workspace_size(M, N, dtype)
    ws = torch.empty(wsz, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(6):
        dx = torch.empty_like(xt)
        dg = torch.empty_like(gt)
        assert B.rmsnorm_bwd(dyt, xt, gt, r, dx, dg, M, N, dtype, 0, ws, wsz) == 0
        outs.append((dx, dg))
    torch.cuda.synchronize()
    for dx, dg in outs[1:]:
        assert torch.equal(dx.view(torch.int16), outs[0][0].view(torch.int16))
        assert torch.equal(dg.view(torch.int16), outs[0][1].view(torch.int16))
    _gate(x, g, dy, dtype, False, (B.to_numpy(y, dtype).reshape(M, N), B.to_numpy(r, "float32"),
                                    B.to_numpy(outs[-1][0], dtype).reshape(M, N), B.to_numpy(outs[-1][1], dtype)),
          "reused workspace")


def test_small_workspace_takes_the_static_assignment():
    """A workspace that holds one partial row per CTA but not the pool's rows (the
    static-scratch entry point's situation) runs the static assignment."""
    from rmsnorm_fwd_bwd_gb300 import binding as B
    M, N, dtype = BASE
    plan = _plan(M, N, dtype)
    assert "pool_head=" in plan
    units = int(dict(kv.split("=") for kv in plan.split()[1:])["units"])
    small = units * N * 4
    assert small < B.rmsnorm_bwd_workspace_size(M, N, dtype)
    x, g, dy = inputs.make_inputs(M, N, dtype, seed=13)
    _gate(x, g, dy, dtype, False, gpu_util.run(x, g, dy, dtype, ws_bytes=small), "static fallback")
    # one byte less than that: rejected before any launch
    with pytest.raises(AssertionError, match="workspace"):
        gpu_util.run(x, g, dy, dtype, ws_bytes=small - 1)


def test_pool_backward_replayed_from_a_cuda_graph():
    """A captured forward + backward repeats the same call tickets on every replay;
    the forward's CTA 0 reopens its queue word and the backward's column reduce
    closes its own after each call, so every replay (with new inputs copied into
    the captured buffers) gives the eager bits."""
    torch = pytest.importorskip("torch")
    from rmsnorm_fwd_bwd_gb300 import binding as B
    M, N, dtype = BASE
    assert "pool_head=" in _plan(M, N, dtype)
    dev = [tuple(B.to_device(a.reshape(-1), dtype) for a in inputs.make_inputs(M, N, dtype, seed=40 + i))
           for i in range(3)]
    x, g, dy = (torch.empty_like(t) for t in dev[0])
    y = torch.empty_like(x)
    r = torch.empty(M, dtype=torch.float32, device="cuda")
    dx = torch.empty_like(x)
    dg = torch.empty_like(g)
    wsz = B.rmsnorm_bwd_workspace_size(M, N, dtype)
    ws = torch.empty(wsz, dtype=torch.uint8, device="cuda")

    def step():
        assert B.rmsnorm_fwd(x, g, y, r, M, N, 1e-6, dtype, 0) == 0
        assert B.rmsnorm_bwd(dy, x, g, r, dx, dg, M, N, dtype, 0, ws, wsz) == 0

    def load(k):
        for dst, src in zip((x, g, dy), dev[k]):
            dst.copy_(src)

    refs = []
    for k in range(len(dev)):
        load(k)
        step()
        torch.cuda.synchronize()
        refs.append((dx.clone(), dg.clone(), y.clone(), r.clone()))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(2):
        for k, (rdx, rdg, ry, rr) in enumerate(refs):
            load(k)
            graph.replay()
            torch.cuda.synchronize()
            assert torch.equal(y.view(torch.int16), ry.view(torch.int16)), f"y differs on replay {k}"
            assert torch.equal(r, rr), f"rstd differs on replay {k}"
            assert torch.equal(dx.view(torch.int16), rdx.view(torch.int16)), f"dx differs on replay {k}"
            assert torch.equal(dg.view(torch.int16), rdg.view(torch.int16)), f"dgamma differs on replay {k}"


@pytest.mark.parametrize("M,N,dtype,offset", [(10000, 4096, "bfloat16", False), (12000, 2048, "float16", True),
                                              (10000, 2048, "float32", False), (4096, 4096, "bfloat16", True)])
def test_forward_pool_matches_static_and_every_cta_running_every_segment(M, N, dtype, offset):
    """y and r of a row do not depend on which CTA computed it: the forward pool,
    the static assignment, and the pool with its queue bypassed (every CTA runs
    every queued segment, the path of a forward whose queue word is not its own)
    give the same bits; the pool's result is gated against the oracle."""
    from rmsnorm_fwd_bwd_gb300 import binding as B
    plan = B.rmsnorm_describe_plan(0, M, N, dtype)
    if "pool_head=" not in plan:
        pytest.skip(f"no row pool in this plan: {plan}")
    x, g, dy = inputs.make_inputs(M, N, dtype, seed=M + 3 * N, offset=offset)
    outs = {}
    try:
        for mode in (1, 0, 2):
            assert B.rmsnorm_set_row_pool(mode) == 0
            y, r, _, _ = gpu_util.run(x, g, dy, dtype, offset=offset, do_bwd=False)
            outs[mode] = (y, r)
    finally:
        assert B.rmsnorm_set_row_pool(1) == 0
    for mode in (0, 2):
        assert np.array_equal(outs[mode][0], outs[1][0]) and np.array_equal(outs[mode][1], outs[1][1]), mode
    res = check.gate_outputs(x, g, dy, dtype, offset, 1e-6, y=outs[1][0], rstd=outs[1][1])
    text = gate.report(f"forward pool {plan}", res)
    print("\n" + text)
    assert gate.overall(res) == "PASS", text
