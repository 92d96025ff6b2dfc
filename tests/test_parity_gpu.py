"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Every case gates y, rstd, dx and dgamma with the golden / reference / target
gate (constants in oracle/gate.py, declared before any run). Shapes follow the
torchtitan page's tile-boundary table and adversarial variance cases, the
printed worked examples, and the measured workloads (full size where the
oracle finishes in seconds, sampled rows otherwise).
"""
import numpy as np
import pytest

from oracle import check, gate
from oracle import oracle as orc
from rmsnorm_fwd_bwd_gb300 import inputs

from . import gpu_util, row_threads

pytestmark = pytest.mark.gpu

DTYPES = ["float32", "float16", "bfloat16"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rmsnorm_fwd_bwd_gb300 import binding
    binding.rmsnorm_device_error(clear=True)
    yield
    assert binding.rmsnorm_device_error(clear=True) == 0, "a kernel reported a wait timeout"


def _assert_pass(results, title, allow_limited=False):
    text = gate.report(title, results)
    print("\n" + text)
    ok = ("PASS", "PASS WITH LIMITATIONS") if allow_limited else ("PASS",)
    assert gate.overall(results) in ok, text


def _gate_case(x, g, dy, dtype, offset=False, eps=1e-6, misalign=False, title="", row_groups=None,
               allow_limited=False):
    y, r, dx, dg = gpu_util.run(x, g, dy, dtype, offset=offset, eps=eps, misalign=misalign)
    res = check.gate_outputs(x, g, dy, dtype, offset, eps, y=y, rstd=r, dx=dx, dgamma=dg,
                             row_groups=row_groups)
    _assert_pass(res, title or f"{dtype} {x.shape} offset={offset} misalign={misalign}",
                 allow_limited)
    return y, r, dx, dg


# --------------------------------------------------------------------------- #
# printed worked examples
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("dtype", DTYPES)
def test_worked_examples(golden_file, dtype):
    f = golden_file("forward_worked_example.txt")
    b = golden_file("backward_worked_example.txt")
    x = inputs.to_storage(np.array([f["x"][0]], np.float32), dtype)
    dy = inputs.to_storage(np.array([b["dy"][0]], np.float32), dtype)
    uo = {"float32": 2 ** -24, "float16": 2 ** -11, "bfloat16": 2 ** -8}[dtype]
    for gk, yk in (("gamma", "y"), ("gamma_b", "y_b")):
        g = inputs.to_storage(np.array(f[gk][0], np.float32), dtype)
        y, r, dx, dg = _gate_case(x, g, dy, dtype, title=f"worked example {gk} {dtype}")
        yv = orc.decode(y, dtype)[0]
        for got, want, d in zip(yv, *f[yk]):
            assert abs(got - want) <= 0.5 * 10 ** -d + abs(want) * uo
        assert abs(r[0] - f["r"][0][0]) <= 0.5e-6
        if gk == "gamma":
            dxv = orc.decode(dx, dtype)[0]
            for got, want, d in zip(dxv, *b["dx"]):
                assert abs(got - want) <= 0.5 * 10 ** -d + abs(want) * uo


# --------------------------------------------------------------------------- #
# tile-boundary shapes and adversarial variance (torchtitan page's case table)
# --------------------------------------------------------------------------- #
SHAPES = [((3, 255), "float32"), ((3, 256), "bfloat16"), ((3, 257), "bfloat16"),
          ((3, 257), "float16"), ((48, 256), "bfloat16"), ((8, 4095), "bfloat16"),
          ((8, 4096), "bfloat16"), ((8, 4097), "bfloat16"), ((8, 5120), "bfloat16"),
          # rows off 16 bytes: the ragged TMA ring (bf16, fp16 and fp32 up to 16 KB)
          # and the row-vector kernels (rows of 16-20 KB)
          ((29, 4099), "float32"), ((31, 4097), "float16"), ((33, 9999), "bfloat16"),
          # 16-32 KB rows: the backward's one-block (up to 512 threads) plans
          ((5, 16384), "float16"), ((7, 8192), "float32"), ((3, 10240), "bfloat16")]


@pytest.mark.parametrize("shape,dtype", SHAPES)
@pytest.mark.parametrize("offset", [False, True])
def test_tile_boundary_shapes(shape, dtype, offset):
    M, N = shape
    x, g, dy = inputs.make_inputs(M, N, dtype, seed=M * 131 + N, offset=offset)
    _gate_case(x, g, dy, dtype, offset=offset)


@pytest.mark.parametrize("scale", [1e-5, 0.0])
def test_near_zero_and_zero_variance(scale):
    M, N, dtype = 8, 5120, "bfloat16"
    x, g, dy = inputs.make_inputs(M, N, dtype, seed=9, x_scale=scale)
    _gate_case(x, g, dy, dtype, title=f"variance scale {scale}")


@pytest.mark.parametrize("M", [1, 17])
def test_dgamma_sum_over_rows(M):
    x, g, dy = inputs.make_inputs(M, 384, "float32", seed=M)
    _gate_case(x, g, dy, "float32", title=f"M={M}")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("N", [1, 2, 3, 7, 8, 33, 1000, 16384])
def test_small_and_max_widths(dtype, N):
    M = 37 if N <= 1000 else 9
    x, g, dy = inputs.make_inputs(M, N, dtype, seed=N)
    # N = 1 is the degenerate width: dx = r*u*eps/(x^2+eps) cancels almost entirely
    _gate_case(x, g, dy, dtype, allow_limited=(N == 1))


@pytest.mark.parametrize("dtype,N", [("bfloat16", 4096), ("float32", 16384), ("float16", 8192),
                                     ("bfloat16", 5120)])
@pytest.mark.parametrize("offset", [False, True])
def test_misaligned_pointers_take_general_path(dtype, N, offset):
    M = 65
    x, g, dy = inputs.make_inputs(M, N, dtype, seed=5, offset=offset)
    _gate_case(x, g, dy, dtype, offset=offset, misalign=True)


@pytest.mark.parametrize("names", [("y",), ("dx",), ("y", "dx"), ("dy",), ("x",), ("g",)])
@pytest.mark.parametrize("dtype,N", [("bfloat16", 4096), ("bfloat16", 4099), ("float32", 1023)])
def test_partially_misaligned_tensors(names, dtype, N):
    """Outputs at another 16-byte phase than x (element stores at every vector),
    and x/dy at different phases (general scalar path)."""
    x, g, dy = inputs.make_inputs(37, N, dtype, seed=len(names) + N)
    _gate_case(x, g, dy, dtype, misalign=set(names), title=f"{dtype} N={N} shifted={names}")


def test_many_rows_narrow():
    for M, N, dtype in ((100003, 64, "float32"), (50001, 8, "bfloat16"), (20011, 24, "float16")):
        x, g, dy = inputs.make_inputs(M, N, dtype, seed=3)
        _gate_case(x, g, dy, dtype)


# --------------------------------------------------------------------------- #
# the measured workloads
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("name", ["fp32_64x256", "bf16_4096x4096", "bf16_adversarial_8192x5120",
                                  "bf16_adversarial_8192x4099"])
def test_workload_full(name):
    w = inputs.WORKLOADS[name]
    x, g, dy = inputs.workload_inputs(w)
    groups = None
    if w.adversarial:
        cls = np.arange(w.M) % 5
        groups = {f"class{c}": np.nonzero(cls == c)[0] for c in range(5)}
    _gate_case(x, g, dy, w.dtype, offset=w.offset, eps=w.eps, title=name, row_groups=groups)


@pytest.mark.parametrize("name", ["fp16_offset_16384x8192", "fp16_offset_16384x16384",
                                  "fp32_offset_16384x8192", "fp32_offset_16384x16384"])
def test_wide_rows_cluster_path(name):
    """The cluster (DSMEM) path at the workloads' widths, on a ragged row count."""
    w = inputs.WORKLOADS[name]
    x, g, dy = inputs.make_inputs(515, w.N, w.dtype, seed=1, offset=w.offset)
    _gate_case(x, g, dy, w.dtype, offset=w.offset, eps=w.eps, title=f"{name} rows=515")


@pytest.mark.parametrize("name", ["bf16_65536x4096", "fp16_offset_16384x16384",
                                  "fp32_offset_16384x16384", "fp16_offset_16384x8192",
                                  "fp32_offset_16384x8192"])
def test_workload_full_size_every_row(name):
    """Full-size launch in the benchmark's configuration, gated on every row:
    y, rstd and dx of all M rows and dgamma over all of them. The oracle's
    per-row functions run over row chunks in parallel threads (each row is
    computed on its own, so the values are those of one call). dgamma must also
    pass the gate built on the pairwise-summed fp32 reference: these M >= 8192
    sums are where a sequential reference is least accurate, and the kernel's
    blocked sum must not need that slack."""
    w = inputs.WORKLOADS[name]
    x, g, dy = inputs.workload_inputs(w)
    y, r, dx, dg = gpu_util.run(x, g, dy, w.dtype, offset=w.offset, eps=w.eps)
    res = check.gate_outputs(x, g, dy, w.dtype, w.offset, w.eps, y=y, rstd=r, dx=dx, dgamma=dg,
                             map_rows=row_threads.map_rows)
    _assert_pass(res, f"{name} (every row)")
    dgr = [q for q in res if q.tensor == "dgamma"][0]
    assert dgr.pairwise_within, dgr.notes


# --------------------------------------------------------------------------- #
# determinism, empty inputs, errors, dispatch
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("name", ["bf16_4096x4096", "bf16_adversarial_8192x4099"])
def test_repeated_runs_are_bitwise_identical(name):
    w = inputs.WORKLOADS[name]
    x, g, dy = inputs.workload_inputs(w)
    first = gpu_util.run(x, g, dy, w.dtype, offset=w.offset)
    for _ in range(2):
        again = gpu_util.run(x, g, dy, w.dtype, offset=w.offset)
        for a, b in zip(first, again):
            assert np.array_equal(a, b)


def test_empty_rows():
    import torch
    from rmsnorm_fwd_bwd_gb300 import binding as B
    N = 300
    g = torch.randn(N, device="cuda")
    dg = torch.full((N,), 7.0, device="cuda")
    e = torch.empty(0, device="cuda")
    assert B.rmsnorm_fwd(e, g, e, e, 0, N, 1e-6, "float32", 0) == B.RMSNORM_OK
    assert B.rmsnorm_bwd_workspace_size(0, N, "float32") == 0
    assert B.rmsnorm_bwd(e, e, g, e, e, dg, 0, N, "float32", 0, None, 0) == B.RMSNORM_OK
    torch.cuda.synchronize()
    assert torch.all(dg == 0)


def test_rejections_write_nothing():
    import torch
    from rmsnorm_fwd_bwd_gb300 import binding as B
    M, N = 64, 512
    x = torch.randn(M, N, device="cuda", dtype=torch.bfloat16)
    g = torch.ones(N, device="cuda", dtype=torch.bfloat16)
    y = torch.full_like(x, 3.0)
    r = torch.full((M,), 5.0, device="cuda")
    assert B.rmsnorm_fwd(x, g, y, r, M, 16385, 1e-6, "bfloat16", 0) == 2          # SHAPE
    assert B.rmsnorm_fwd(x, g, y, r, M, N, 0.0, "bfloat16", 0) == 4               # EPS
    assert B.rmsnorm_fwd(x, g, y, r, M, N, float("nan"), "bfloat16", 0) == 4
    assert B.rmsnorm_fwd(x, g, y, r, M, N, 1e-6, 7, 0) == 3                       # DTYPE
    assert B.rmsnorm_fwd(x, g, y, r, M, N, 1e-6, "bfloat16", 2) == 9              # ARG
    assert B.rmsnorm_fwd(x.data_ptr() + 1, g, y, r, M, N, 1e-6, "bfloat16", 0) == 5  # ALIGN
    dx = torch.full_like(x, 3.0)
    dg = torch.full_like(g, 3.0)
    need = B.rmsnorm_bwd_workspace_size(M, N, "bfloat16")
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    # the size query covers every layout's plan; one row of partials (N floats) is
    # less than any plan needs
    assert B.rmsnorm_bwd(x, x, g, r, dx, dg, M, N, "bfloat16", 0, ws, N * 4 - 16) == 6  # WORKSPACE
    assert B.rmsnorm_bwd(x, x, g, r, dx, dg, M, N, "bfloat16", 0, None, need) == 1     # NULL
    torch.cuda.synchronize()
    assert torch.all(y == 3.0) and torch.all(r == 5.0)
    assert torch.all(dx == 3.0) and torch.all(dg == 3.0)


def test_plan_dispatch():
    from rmsnorm_fwd_bwd_gb300 import binding as B
    assert B.rmsnorm_describe_plan(0, 65536, 4096, "bfloat16").startswith("tma cluster=1")
    assert B.rmsnorm_describe_plan(1, 65536, 4096, "bfloat16").startswith("tma cluster=1")
    assert B.rmsnorm_describe_plan(0, 16384, 16384, "float32").startswith("tma cluster=4")
    # 32 KB rows stay in one block: 256 threads x 8 vectors forward, 512 x 4 backward
    assert B.rmsnorm_describe_plan(0, 16384, 16384, "float16").startswith("tma cluster=1 threads=256 vpt=8")
    assert B.rmsnorm_describe_plan(1, 16384, 16384, "float16").startswith("tma cluster=1 threads=512 vpt=4")
    assert B.rmsnorm_describe_plan(1, 16384, 8192, "float32").startswith("tma cluster=1 threads=512 vpt=4")
    assert B.rmsnorm_describe_plan(1, 16384, 16384, "float32").startswith("tma cluster=4")
    assert B.rmsnorm_describe_plan(0, 8192, 4099, "bfloat16").startswith("ragged")
    assert B.rmsnorm_describe_plan(1, 8192, 4099, "bfloat16").startswith("ragged")
    assert B.rmsnorm_describe_plan(0, 8192, 4096, "bfloat16", aligned16=False).startswith("ragged")
    assert B.rmsnorm_describe_plan(1, 29, 4099, "float32").startswith("ragged")
    assert B.rmsnorm_describe_plan(0, 33, 9999, "bfloat16").startswith("rowvec")
    assert B.rmsnorm_describe_plan(1, 33, 9999, "bfloat16").startswith("rowvec")
    assert B.rmsnorm_describe_plan(1, 8192, 4096, "bfloat16", aligned16=2).startswith("scalar")
    assert B.rmsnorm_describe_plan(0, 64, 16383, "float32", aligned16=False).startswith("scalar")

    def blocks_per_sm(plan):
        f = dict(kv.split("=") for kv in plan.split()[1:])
        return int(f["units"]) / int(f["sms"])
    # backward with few rows per SM: as many blocks as fit, up to 4 (smem caps
    # 20 KB rows at 3); many rows per SM: the 96 KB ring target (3 at 8 KB rows)
    assert blocks_per_sm(B.rmsnorm_describe_plan(1, 4096, 4096, "bfloat16")) == 4
    assert blocks_per_sm(B.rmsnorm_describe_plan(1, 8192, 5120, "bfloat16")) == 3
    assert blocks_per_sm(B.rmsnorm_describe_plan(1, 65536, 4096, "bfloat16")) == 3


def test_torch_conveniences_match_raw_calls():
    import torch
    from rmsnorm_fwd_bwd_gb300 import binding as B
    x, g, dy = inputs.make_inputs(33, 768, "bfloat16", seed=4)
    xt, gt, dyt = (B.to_device(a, "bfloat16") for a in (x, g, dy))
    y, r = B.forward(xt.view(33, 768), gt)
    dx, dg = B.backward(dyt.view(33, 768), xt.view(33, 768), gt, r)
    ref = gpu_util.run(x, g, dy, "bfloat16")
    assert np.array_equal(B.to_numpy(y, "bfloat16").reshape(33, 768), ref[0])
    assert np.array_equal(B.to_numpy(r, "float32"), ref[1])
    assert np.array_equal(B.to_numpy(dx, "bfloat16").reshape(33, 768), ref[2])
    assert np.array_equal(B.to_numpy(dg, "bfloat16"), ref[3])
