"""GPU parity of the LayerNorm kernels (layernorm_fwd / layernorm_bwd) against
the CPU oracle.

Every case gates y, mean, rstd, dx, dgamma and dbeta with the golden /
reference / target gate. Shapes cover the TMA path (one CTA per row slice),
the cluster path (rows split over 2 and 4 CTAs), the ragged TMA path (rows off
16 bytes up to 16 KB), the row-vector path (such rows of 16-20 KB), the general path (rows over 20 KB that are not 16-byte
multiples, x and dy at different 16-byte phases), tiny and empty inputs, rows with a large mean (where a
one-pass variance would cancel), constant rows (variance 0), strided rows, and
the measured LayerNorm workloads at full size on sampled rows.
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


def _assert_pass(results, title, allow_limited=False):
    text = gate.report(title, results)
    print("\n" + text)
    ok = ("PASS", "PASS WITH LIMITATIONS") if allow_limited else ("PASS",)
    assert gate.overall(results) in ok, text


def _gate(x, g, b, dy, dtype, eps=1e-5, misalign=False, title="", allow_limited=False):
    y, mean, rstd, dx, dg, db = gpu_util.ln_run(x, g, b, dy, dtype, eps=eps, misalign=misalign)
    res = check.gate_ln_outputs(x, g, b, dy, dtype, eps, y=y, mean=mean, rstd=rstd, dx=dx, dgamma=dg,
                                dbeta=db)
    _assert_pass(res, title or f"layernorm {dtype} {x.shape} misalign={misalign}", allow_limited)
    return y, mean, rstd, dx, dg, db


def _plan(pass_, M, N, dtype, aligned16=1):
    """aligned16: 1 aligned, 0 x and dy at one shared 16-byte phase, 2 different phases."""
    from rmsnorm_fwd_bwd_gb300 import binding as B
    return B.rmsnorm_describe_plan(pass_, M, N, dtype, aligned16)


# (dtype, M, N, expected path prefix of the forward plan)
SHAPES = [
    ("float32", 64, 256, "lanes"),
    ("bfloat16", 300, 4096, "tma cluster=1"),
    ("float16", 129, 1000, "lanes"),
    ("bfloat16", 77, 8, "lanes"),
    ("bfloat16", 65, 2048, "tma cluster=1"),
    ("float32", 41, 8192, "tma cluster=2"),
    ("bfloat16", 40, 16384, "tma cluster=2"),
    ("float16", 33, 12288, "tma cluster=2"),
    ("float32", 24, 16384, "tma cluster=4"),
    ("bfloat16", 67, 4099, "ragged"),
    ("float32", 50, 333, "ragged"),
    ("float32", 29, 4099, "ragged"),
    ("float16", 31, 9999, "rowvec"),
    ("float32", 29, 6001, "scalar"),
    ("bfloat16", 23, 16383, "scalar"),
]


@pytest.mark.parametrize("dtype,M,N,path", SHAPES)
def test_shapes_and_paths(dtype, M, N, path):
    assert _plan(2, M, N, dtype).startswith(path)
    assert _plan(3, M, N, dtype).startswith(path)
    x, g, b, dy = inputs.make_ln_inputs(M, N, dtype, seed=N + M)
    _gate(x, g, b, dy, dtype, title=f"layernorm {dtype} {M}x{N} ({path})")


@pytest.mark.parametrize("dtype", ["float32", "float16", "bfloat16"])
def test_misaligned_pointers(dtype):
    # all tensors one element off (row-vector path, outputs at the rows' phase);
    # only the outputs off (row-vector path, element stores); x off but dy not
    # (the backward's general path)
    M, N = 45, 2048
    assert _plan(2, M, N, dtype, 0).startswith("ragged") and _plan(3, M, N, dtype, 0).startswith("ragged")
    assert _plan(3, M, N, dtype, 2).startswith("scalar")
    x, g, b, dy = inputs.make_ln_inputs(M, N, dtype, seed=11)
    _gate(x, g, b, dy, dtype, misalign=True, title=f"layernorm {dtype} misaligned")
    _gate(x, g, b, dy, dtype, misalign={"y", "dx"}, title=f"layernorm {dtype} misaligned outputs")
    _gate(x, g, b, dy, dtype, misalign={"x"}, title=f"layernorm {dtype} x and dy at different phases")


@pytest.mark.parametrize("N", [1, 2, 3])
def test_tiny_rows(N):
    # N = 1: variance 0, y = beta, dx = 0. N = 2: x_hat = +-1 up to eps, and dx
    # is only what eps leaves of terms that cancel exactly without it; there the
    # fp32 reference itself misses the fp32 normwise bound, so the gate's
    # "PASS WITH LIMITATIONS" (main gate passed, bound not attainable) is accepted.
    x, g, b, dy = inputs.make_ln_inputs(19, N, "float32", seed=N)
    y, mean, rstd, dx, dg, db = _gate(x, g, b, dy, "float32", title=f"layernorm N={N}",
                                      allow_limited=N == 2)
    if N == 1:
        assert np.array_equal(y, np.tile(b, (19, 1)))
        assert np.all(dx == 0)


@pytest.mark.parametrize("dtype,N", [("bfloat16", 4096), ("float32", 16384), ("float16", 3000)])
def test_large_row_means(dtype, N):
    """Rows whose mean is far larger than their spread: a variance formed as
    mean(x^2) - mean(x)^2 would lose most of its digits here."""
    M = 48
    xs = inputs.normal(5, 0, (M, N)) + np.float32(200.0) + inputs.normal(5, 5, (M, 1), 30.0)
    _, g, b, dy = inputs.make_ln_inputs(M, N, dtype, seed=5)
    x = inputs.to_storage(xs, dtype)
    _gate(x, g, b, dy, dtype, title=f"layernorm {dtype} N={N} large means")


@pytest.mark.parametrize("dtype,N", [("bfloat16", 4096), ("float32", 8192), ("float16", 1001), ("float16", 1000)])
def test_constant_rows(dtype, N):
    # values on a 1/16 grid: every partial sum is exact, so the mean is the row's
    # value, x_hat = 0 exactly, y = beta and dgamma = 0
    M = 20
    xs = np.round(np.repeat(inputs.normal(6, 0, (M, 1), 3.0), N, axis=1) * 16) / 16
    xs[::3] = 0.0
    _, g, b, dy = inputs.make_ln_inputs(M, N, dtype, seed=6)
    x = inputs.to_storage(xs.astype(np.float32), dtype)
    y, mean, rstd, dx, dg, db = _gate(x, g, b, dy, dtype, title=f"layernorm {dtype} constant rows")
    assert np.array_equal(y, np.tile(b, (M, 1)))
    assert np.all(inputs.to_storage(np.zeros(N, np.float32), dtype) == dg)


def test_forward_without_saved_statistics():
    M, N, dtype = 200, 4096, "bfloat16"
    x, g, b, dy = inputs.make_ln_inputs(M, N, dtype, seed=12)
    y0, *_ = gpu_util.ln_run(x, g, b, dy, dtype, do_bwd=False)
    y1, *_ = gpu_util.ln_run(x, g, b, dy, dtype, do_bwd=False, stats=False)
    assert np.array_equal(y0, y1)
    xs, gs, bs, dys = inputs.make_ln_inputs(M, 333, "float32", seed=12)
    z0, *_ = gpu_util.ln_run(xs, gs, bs, dys, "float32", do_bwd=False)
    z1, *_ = gpu_util.ln_run(xs, gs, bs, dys, "float32", do_bwd=False, stats=False)
    assert np.array_equal(z0, z1)


@pytest.mark.parametrize("dtype,N", [("bfloat16", 4096), ("float32", 16384), ("bfloat16", 4099)])
def test_repeated_runs_are_bitwise_identical(dtype, N):
    x, g, b, dy = inputs.make_ln_inputs(700, N, dtype, seed=13)
    first = gpu_util.ln_run(x, g, b, dy, dtype)
    again = gpu_util.ln_run(x, g, b, dy, dtype)
    for a, c in zip(first, again):
        assert np.array_equal(a, c)


def test_empty_rows_zero_the_column_gradients():
    import torch
    from rmsnorm_fwd_bwd_gb300 import binding as B
    N = 300
    g = torch.randn(N, device="cuda")
    dg = torch.full((N,), 7.0, device="cuda")
    db = torch.full((N,), 7.0, device="cuda")
    e = torch.empty(0, device="cuda")
    assert B.layernorm_fwd(e, N, g, g, e, N, e, e, 0, N, 1e-5, "float32") == B.RMSNORM_OK
    assert B.layernorm_bwd_workspace_size(0, N, "float32") == 0
    assert B.layernorm_bwd(e, N, e, N, g, e, e, e, N, dg, db, 0, N, "float32", None, 0) == B.RMSNORM_OK
    torch.cuda.synchronize()
    assert torch.all(dg == 0) and torch.all(db == 0)


SENT = {"float32": -12345.5, "float16": 1234.0, "bfloat16": 1234.0}


@pytest.mark.parametrize("dtype,N,ldx,lddy,ldo", [
    ("bfloat16", 4096, 4160, 4160, 4160),      # TMA path with pitches
    ("float32", 8192, 8200, 8204, 8196),       # cluster path with pitches
    ("bfloat16", 4096, 4100, 4100, 4100),      # pitches off 16 bytes: general path
    ("float16", 1000, 1003, 1007, 1024),
])
def test_strided_rows(dtype, N, ldx, lddy, ldo):
    import torch
    from rmsnorm_fwd_bwd_gb300 import binding as B
    M = 67
    x, g, b, dy = inputs.make_ln_inputs(M, N, dtype, seed=N + ldx)
    tdt = getattr(torch, dtype)

    def wide(a, ld):
        buf = torch.full((M, ld), SENT[dtype], dtype=tdt, device="cuda")
        buf[:, :N] = B.to_device(a.reshape(-1), dtype).view(M, N)
        return buf

    xb, dyb = wide(x, ldx), wide(dy, lddy)
    gt, bt = B.to_device(g, dtype), B.to_device(b, dtype)
    yb = torch.full((M, ldo), SENT[dtype], dtype=tdt, device="cuda")
    dxb = torch.full((M, ldo), SENT[dtype], dtype=tdt, device="cuda")
    mean = torch.empty(M, device="cuda")
    rstd = torch.empty(M, device="cuda")
    dg, db = torch.empty_like(gt), torch.empty_like(bt)
    assert B.layernorm_fwd(xb, ldx, gt, bt, yb, ldo, mean, rstd, M, N, 1e-5, dtype) == 0
    need = B.layernorm_bwd_workspace_size(M, N, dtype)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    assert B.layernorm_bwd(dyb, lddy, xb, ldx, gt, mean, rstd, dxb, ldo, dg, db, M, N, dtype, ws, need) == 0
    torch.cuda.synchronize()
    for buf in (yb, dxb):
        assert torch.all(buf[:, N:] == SENT[dtype]), "a gap element between rows was written"
    res = check.gate_ln_outputs(x, g, b, dy, dtype, 1e-5,
                                y=B.to_numpy(yb[:, :N].contiguous(), dtype),
                                mean=B.to_numpy(mean, "float32"), rstd=B.to_numpy(rstd, "float32"),
                                dx=B.to_numpy(dxb[:, :N].contiguous(), dtype),
                                dgamma=B.to_numpy(dg, dtype), dbeta=B.to_numpy(db, dtype))
    _assert_pass(res, f"layernorm strided {dtype} N={N} ld={ldx},{lddy},{ldo}")


def test_rejections_write_nothing():
    import torch
    from rmsnorm_fwd_bwd_gb300 import binding as B
    M, N = 64, 512
    x = torch.randn(M, N, device="cuda", dtype=torch.bfloat16)
    g = torch.ones(N, device="cuda", dtype=torch.bfloat16)
    y = torch.full_like(x, 3.0)
    m = torch.full((M,), 5.0, device="cuda")
    r = torch.full((M,), 5.0, device="cuda")
    assert B.layernorm_fwd(x, N, g, g, y, N, m, r, M, 16385, 1e-5, "bfloat16") == 2
    assert B.layernorm_fwd(x, N, g, g, y, N, m, r, M, N, 0.0, "bfloat16") == 4
    assert B.layernorm_fwd(x, N, g, None, y, N, m, r, M, N, 1e-5, "bfloat16") == 1
    assert B.layernorm_fwd(x.data_ptr() + 1, N, g, g, y, N, m, r, M, N, 1e-5, "bfloat16") == 5
    dx = torch.full_like(x, 3.0)
    dg = torch.full_like(g, 3.0)
    db = torch.full_like(g, 3.0)
    need = B.layernorm_bwd_workspace_size(M, N, "bfloat16")
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    # the size query covers every layout's plan; one row of each plane of partials
    # is less than any plan needs
    assert B.layernorm_bwd(x, N, x, N, g, m, r, dx, N, dg, db, M, N, "bfloat16", ws, 2 * N * 4 - 16) == 6
    assert B.layernorm_bwd(x, N, x, N, g, None, r, dx, N, dg, db, M, N, "bfloat16", ws, need) == 1
    torch.cuda.synchronize()
    assert torch.all(y == 3.0) and torch.all(m == 5.0) and torch.all(r == 5.0)
    assert torch.all(dx == 3.0) and torch.all(dg == 3.0) and torch.all(db == 3.0)


# --------------------------------------------------------------------------- #
# the measured LayerNorm workloads
# --------------------------------------------------------------------------- #
def _sample_rows(M, k=192, seed=0):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([np.arange(32), np.arange(M - 32, M), rng.choice(M, k, replace=False)]))


@pytest.mark.parametrize("name", ["ln_bf16_65536x4096", "ln_fp32_16384x16384", "ln_bf16_16384x4099"])
def test_workload_full_size_sampled(name):
    """Full-size launch (the benchmark's configuration): y, mean, rstd and dx
    gated on sampled rows, dgamma and dbeta gated in full."""
    w = inputs.WORKLOADS[name]
    x, g, b, dy = inputs.workload_inputs(w)
    y, mean, rstd, dx, dg, db = gpu_util.ln_run(x, g, b, dy, w.dtype, eps=w.eps)
    rows = _sample_rows(w.M)
    res = check.gate_ln_outputs(x, g, b, dy, w.dtype, w.eps, y=y[rows], mean=mean[rows], rstd=rstd[rows],
                                dx=dx[rows], dgamma=dg, dbeta=db, rows=rows)
    _assert_pass(res, f"{name} (sampled rows, full dgamma and dbeta)")
