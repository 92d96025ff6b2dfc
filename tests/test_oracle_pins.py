"""Pins of the CPU oracle to facts outside itself (CPU only).

Each test checks the oracle against something it cannot reproduce by
construction: values printed by the pages (tests/golden/*.txt), closed forms,
invariants, finite differences, library routines, or brute force on tiny inputs.
"""
import math

import numpy as np
import pytest

from oracle import oracle as orc
from rmsnorm_fwd_bwd_gb300 import inputs

DTYPES = ["float32", "float16", "bfloat16"]


def _tol(decimals):
    return 0.5 * 10.0 ** (-decimals) + 1e-12


def _store(values, dtype):
    return inputs.to_storage(np.asarray(values, np.float32), dtype)


# --------------------------------------------------------------------------- #
# printed worked examples
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("dtype", DTYPES)
def test_forward_worked_example(golden_file, dtype):
    g = golden_file("forward_worked_example.txt")
    eps = g["eps"][0][0]
    x = _store([g["x"][0]], dtype)
    for gk, yk in (("gamma", "y"), ("gamma_b", "y_b")):
        gam = _store(g[gk][0], dtype)
        y, r = orc.fwd_golden(x, gam, dtype, eps=eps)
        (rv,), (rd,) = g["r"]
        assert abs(r[0] - rv) <= _tol(rd)
        for got, want, d in zip(y[0], *g[yk]):
            assert abs(got - want) <= _tol(d), (gk, got, want)
        # the fp32-intermediate reference reaches the same printed digits
        # (plus the output dtype's own rounding)
        yr, rr = orc.fwd_reference(x, gam, dtype, eps=eps)
        yr = orc.decode(yr, dtype)[0]
        for got, want, d in zip(yr, *g[yk]):
            assert abs(got - want) <= _tol(d) + abs(want) * {"float32": 1e-7, "float16": 2 ** -11,
                                                             "bfloat16": 2 ** -8}[dtype]
    # intermediate steps of the printed table, recomputed from the golden r
    (den,), (dd,) = g["denominator"]
    assert abs(1.0 / r[0] - den) <= _tol(dd)


@pytest.mark.parametrize("dtype", DTYPES)
def test_backward_worked_example(golden_file, dtype):
    g = golden_file("backward_worked_example.txt")
    eps = g["eps"][0][0]
    x = _store([g["x"][0]], dtype)
    gam = _store(g["gamma"][0], dtype)
    dy = _store([g["dy"][0]], dtype)
    dx, dg = orc.bwd_golden(dy, x, gam, dtype, eps=eps)
    for got, want, d in zip(dx[0], *g["dx"]):
        assert abs(got - want) <= _tol(d), (got, want)
    # mean(u*x) = 5.5 is exact; with it, dx follows from r alone:
    # dx = r*u - x*r^3*5.5. Check the oracle agrees with that decomposition.
    _, r = orc.fwd_golden(x, gam, dtype, eps=eps)
    u = np.array(g["u"][0])
    xs = np.array(g["x"][0])
    mean_ux = g["mean_ux"][0][0]
    assert mean_ux == float(np.mean(u * xs))
    np.testing.assert_allclose(dx[0], r[0] * u - xs * r[0] ** 3 * mean_ux, rtol=1e-14)
    # dgamma of the same example (derived, not printed): dy * x * r
    np.testing.assert_allclose(dg, np.array(g["dy"][0]) * xs * r[0], rtol=1e-14)


def test_dgamma_is_a_sum_not_a_mean(golden_file):
    g = golden_file("dgamma_sum_table.txt")
    dtype = "float32"
    # Rows of ones make r = 1/sqrt(1 + eps); choose dy so that dy*x*r reproduces
    # the table's per-row contributions (up to fp32 storage of dy).
    eps = 1e-6
    contrib = np.array([g["row0"][0], g["row1"][0]])
    x = np.ones((2, 2), np.float32)
    r = 1.0 / math.sqrt(1.0 + eps)
    dy = (contrib / r).astype(np.float32)
    _, dg = orc.bwd_golden(dy, x, np.ones(2, np.float32), dtype, eps=eps)
    np.testing.assert_allclose(dg, g["sum"][0], atol=1e-6)
    assert np.all(np.abs(dg - np.array(g["mean_wrong"][0])) > 1.0)
    _, dgr = orc.bwd_reference(dy, x, np.ones(2, np.float32), dtype, eps=eps)
    np.testing.assert_allclose(dgr, g["sum"][0], atol=1e-5)
    # M = 1 versus M = 17 identical rows: a sum grows 17-fold, a mean would not
    (m1,), _ = g["rows_same"]
    (m17,), _ = g["rows_differ"]
    xr = inputs.normal(5, 0, (1, 9))
    dyr = inputs.normal(5, 2, (1, 9))
    gam = np.float32(1) + inputs.normal(5, 1, (9,), 0.1)
    _, d1 = orc.bwd_golden(np.repeat(dyr, int(m1), 0), np.repeat(xr, int(m1), 0), gam, dtype)
    _, d17 = orc.bwd_golden(np.repeat(dyr, int(m17), 0), np.repeat(xr, int(m17), 0), gam, dtype)
    np.testing.assert_allclose(d17, 17.0 * d1, rtol=1e-13)


def test_block_denominator_exercise(golden_file):
    g = golden_file("block_denominator_exercise.txt")
    eps = g["eps"][0][0]
    N = int(g["N"][0][0])
    B = int(g["BLOCK"][0][0])
    ones = np.ones((1, N), np.float32)
    y, r = orc.fwd_golden(ones, np.ones(N, np.float32), "float32", eps=eps)
    for key, val in (("y_correct", y[0, 0]), ("denominator_correct", 1.0 / r[0])):
        (want,), (d,) = g[key]
        assert abs(val - want) <= _tol(d), (key, val, want)
    assert np.all(y[0] == y[0, 0])
    # The wrong variant counts the masked padding in the mean. Reproduce it by
    # running the same oracle over the zero-padded BLOCK-wide row.
    padded = np.zeros((1, B), np.float32)
    padded[0, :N] = 1.0
    yw, rw = orc.fwd_golden(padded, np.ones(B, np.float32), "float32", eps=eps)
    for key, val in (("y_wrong", yw[0, 0]), ("denominator_wrong", 1.0 / rw[0])):
        (want,), (d,) = g[key]
        assert abs(val - want) <= _tol(d), (key, val, want)
    assert g["mean_wrong"][0][0] == N / B
    # small row of the same section: mean 1 with N = 3, 0.75 with a 4-wide block
    small = np.array([g["small_row"][0]], np.float32)
    _, rs = orc.fwd_golden(small, np.ones(3, np.float32), "float32", eps=0.0 + 1e-300)
    assert abs(1.0 / rs[0] ** 2 - g["small_mean_correct"][0][0]) < 1e-12
    pad4 = np.array([[1, 1, 1, 0]], np.float32)
    _, r4 = orc.fwd_golden(pad4, np.ones(4, np.float32), "float32", eps=1e-300)
    assert abs(1.0 / r4[0] ** 2 - g["small_mean_wrong"][0][0]) < 1e-12


# --------------------------------------------------------------------------- #
# invariants and closed forms
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("offset", [False, True])
def test_zero_row(dtype, offset):
    N = 33
    x = _store(np.zeros((2, N)), dtype)
    gam = _store(1.0 + 0.1 * inputs.normal(1, 1, (N,)), dtype)
    dy = _store(inputs.normal(1, 2, (2, N)), dtype)
    y, r = orc.fwd_golden(x, gam, dtype, offset=offset)
    assert np.all(y == 0.0)
    np.testing.assert_allclose(r, 1000.0, rtol=1e-12)   # 1/sqrt(1e-6)
    dx, dg = orc.bwd_golden(dy, x, gam, dtype, offset=offset)
    gv = orc.decode(gam, dtype) + (1.0 if offset else 0.0)
    np.testing.assert_allclose(dx, 1000.0 * gv * orc.decode(dy, dtype), rtol=1e-12)
    assert np.all(dg == 0.0)
    yr, rr = orc.fwd_reference(x, gam, dtype, offset=offset)
    assert np.all(orc.decode(yr, dtype) == 0.0)
    np.testing.assert_allclose(rr, 1000.0, rtol=1e-6)


def test_scale_invariance():
    # y(c*x) = y(x) up to the effect of eps: |dy/y| <= eps / (2 mean(x^2)).
    x = inputs.normal(3, 0, (4, 64))
    gam = np.float32(1) + inputs.normal(3, 1, (64,), 0.1)
    y1, r1 = orc.fwd_golden(x, gam, "float32")
    for c in (4.0, 0.25, 1024.0):
        y2, r2 = orc.fwd_golden((x * np.float32(c)).astype(np.float32), gam, "float32")
        ms = np.mean(x.astype(np.float64) ** 2, axis=1, keepdims=True)
        bound = 1e-6 / (2 * ms * min(1.0, c * c)) + 1e-14
        assert np.all(np.abs(y2 - y1) <= bound * np.abs(y1) + 1e-300)
        np.testing.assert_allclose(r2 * c, r1, rtol=float(np.max(bound)))


def test_single_column_closed_form():
    # N = 1: mean(x^2) = x^2, so y = gamma * x / sqrt(x^2 + eps) = gamma*sign(x)*(1 - O(eps/x^2)).
    x = np.array([[3.0], [-0.5], [1e-2], [-7.0]], np.float32)
    gam = np.array([1.5], np.float32)
    y, _ = orc.fwd_golden(x, gam, "float32")
    xs = x.astype(np.float64)[:, 0]
    approx = 1.5 * np.sign(xs)
    assert np.all(np.abs(y[:, 0] - approx) <= 1.5 * 1e-6 / xs ** 2)


def test_forward_matches_library_norm():
    # gamma = 1: y = x / sqrt(||x||^2 / N + eps), ||x|| from LAPACK/BLAS nrm2.
    rng_x = inputs.normal(11, 0, (6, 300), 2.0)
    y, r = orc.fwd_golden(rng_x, np.ones(300, np.float32), "float32")
    norms = np.linalg.norm(rng_x.astype(np.float64), axis=1)
    r_lib = 1.0 / np.sqrt(norms ** 2 / 300 + 1e-6)
    np.testing.assert_allclose(r, r_lib, rtol=1e-14)
    np.testing.assert_allclose(y, rng_x * r_lib[:, None], rtol=1e-14)


@pytest.mark.parametrize("offset", [False, True])
def test_backward_finite_differences(offset):
    """Central differences of L = sum(dy * y) against the golden dx and dgamma.

    Inputs lie on a coarse grid (multiples of 2^-8) so that x +/- h with
    h = 2^-12 is exact in float32 storage.
    """
    M, N = 3, 5
    q = 2.0 ** -8
    x = (np.round(inputs.normal(21, 0, (M, N)) / q) * q).astype(np.float32)
    gam = (np.round((np.float32(1) + inputs.normal(21, 1, (N,), 0.3)) / q) * q).astype(np.float32)
    if offset:
        gam = (gam - np.float32(1)).astype(np.float32)
    dy = inputs.normal(21, 2, (M, N))
    dyd = dy.astype(np.float64)
    h = 2.0 ** -12
    eps = 1e-3   # larger eps so that its term is visible in the derivatives

    def loss(xa, ga):
        y, _ = orc.fwd_golden(xa, ga, "float32", eps=eps, offset=offset)
        return float(np.sum(dyd * y))

    dx, dg = orc.bwd_golden(dy, x, gam, "float32", eps=eps, offset=offset)
    fd_x = np.zeros((M, N))
    for i in range(M):
        for j in range(N):
            xp = x.copy(); xp[i, j] += np.float32(h)
            xm = x.copy(); xm[i, j] -= np.float32(h)
            fd_x[i, j] = (loss(xp, gam) - loss(xm, gam)) / (2 * h)
    fd_g = np.zeros(N)
    for j in range(N):
        gp = gam.copy(); gp[j] += np.float32(h)
        gm = gam.copy(); gm[j] -= np.float32(h)
        fd_g[j] = (loss(x, gp) - loss(x, gm)) / (2 * h)
    np.testing.assert_allclose(dx, fd_x, atol=2e-6 * np.max(np.abs(dx)), rtol=0)
    np.testing.assert_allclose(dg, fd_g, atol=2e-6 * np.max(np.abs(dg)), rtol=0)


def test_backward_projection_identity():
    # sum_j x_j dx_j = r*S - r^3 * (S/N) * sum_j x_j^2 = r*S*eps/(mean(x^2)+eps),
    # with S = sum_j u_j x_j: follows from r^2 = 1/(mean(x^2)+eps).
    eps = 0.25
    x = inputs.normal(31, 0, (4, 40))
    dy = inputs.normal(31, 2, (4, 40))
    gam = np.float32(1) + inputs.normal(31, 1, (40,), 0.2)
    dx, _ = orc.bwd_golden(dy, x, gam, "float32", eps=eps)
    xd = x.astype(np.float64)
    S = np.sum(dy.astype(np.float64) * gam.astype(np.float64) * xd, axis=1)
    ms = np.mean(xd ** 2, axis=1)
    r = 1.0 / np.sqrt(ms + eps)
    lhs = np.sum(xd * dx, axis=1)
    np.testing.assert_allclose(lhs, r * S * eps / (ms + eps), rtol=1e-10,
                               atol=1e-12 * np.max(np.abs(r * S)))


# --------------------------------------------------------------------------- #
# reference (fp32 intermediates): brute force and error bounds
# --------------------------------------------------------------------------- #
def _py_store(values32, dtype):
    return inputs.to_storage(np.asarray(values32, np.float32), dtype)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("offset", [False, True])
def test_reference_brute_force(dtype, offset):
    """Tiny inputs: an independent scalar-by-scalar float32 loop (numpy scalars)."""
    M, N = 3, 7
    f32 = np.float32
    x = inputs.to_storage(inputs.normal(41, 0, (M, N), 1.7), dtype)
    gam = inputs.to_storage((0.05 if offset else 1.0) * inputs.normal(41, 1, (N,)) + (0 if offset else 1), dtype)
    dy = inputs.to_storage(inputs.normal(41, 2, (M, N)), dtype)
    xv = orc.decode(x, dtype).astype(np.float32)
    gv = orc.decode(gam, dtype).astype(np.float32)
    dyv = orc.decode(dy, dtype).astype(np.float32)
    eps = f32(1e-6)
    y_bf = np.zeros((M, N), np.float32)
    dx_bf = np.zeros((M, N), np.float32)
    acc = [f32(0)] * N
    r_bf = np.zeros(M, np.float32)
    with np.errstate(all="ignore"):
        for i in range(M):
            ss = f32(0)
            for j in range(N):
                ss = f32(ss + f32(xv[i, j] * xv[i, j]))
            r = f32(f32(1) / f32(np.sqrt(f32(f32(ss / f32(N)) + eps))))
            r_bf[i] = r
            sux = f32(0)
            for j in range(N):
                g = f32(f32(1) + gv[j]) if offset else gv[j]
                sux = f32(sux + f32(f32(dyv[i, j] * g) * xv[i, j]))
            c = f32(sux / f32(N))
            r3 = f32(f32(r * r) * r)
            for j in range(N):
                g = f32(f32(1) + gv[j]) if offset else gv[j]
                y_bf[i, j] = f32(f32(g * xv[i, j]) * r) if offset else f32(f32(xv[i, j] * r) * g)
                u = f32(dyv[i, j] * g)
                dx_bf[i, j] = f32(f32(r * u) - f32(f32(xv[i, j] * r3) * c))
                acc[j] = f32(acc[j] + f32(f32(dyv[i, j] * xv[i, j]) * r))
    y, rstd = orc.fwd_reference(x, gam, dtype, offset=offset)
    dx, dg = orc.bwd_reference(dy, x, gam, dtype, offset=offset)
    np.testing.assert_array_equal(rstd, r_bf)
    np.testing.assert_array_equal(y, _py_store(y_bf, dtype))
    np.testing.assert_array_equal(dx, _py_store(dx_bf, dtype))
    np.testing.assert_array_equal(dg, _py_store(np.array(acc, np.float32), dtype))


@pytest.mark.parametrize("dtype", DTYPES)
def test_reference_close_to_golden(dtype):
    # Standard fp32 error analysis: each output is within (output rounding) +
    # k * u32 * |value|, with k small (a few operations plus the reduction error
    # of a sum of N positive terms, N*u32 relative).
    M, N = 16, 512
    x, gam, dy = inputs.make_inputs(M, N, dtype, seed=7)
    yg, rg = orc.fwd_golden(x, gam, dtype)
    yr, rr = orc.fwd_reference(x, gam, dtype)
    u32 = 2.0 ** -24
    uo = {"float32": 2.0 ** -24, "float16": 2.0 ** -11, "bfloat16": 2.0 ** -8}[dtype]
    assert np.all(np.abs(rr - rg) <= (N + 8) * u32 * rg)
    yrv = orc.decode(yr, dtype)
    assert np.all(np.abs(yrv - yg) <= (uo + (N + 16) * u32) * np.abs(yg) + 1e-30)
    dxg, dgg = orc.bwd_golden(dy, x, gam, dtype)
    dxr, dgr = orc.bwd_reference(dy, x, gam, dtype)
    # dx has cancellation; bound it normwise per row by |r*u| + |x r^3 c| magnitudes
    xv, dyv, gv = orc.decode(x, dtype), orc.decode(dy, dtype), orc.decode(gam, dtype)
    r = rg[:, None]
    c = np.mean(dyv * gv * xv, axis=1, keepdims=True)
    mag = np.abs(r * dyv * gv) + np.abs(xv * r ** 3 * c)
    cmag = np.abs(xv * r ** 3) * np.mean(np.abs(dyv * gv * xv), axis=1, keepdims=True)
    bound = uo * np.abs(dxg) + 16 * u32 * mag + (N + 8) * u32 * cmag
    assert np.all(np.abs(orc.decode(dxr, dtype) - dxg) <= bound + 1e-30)
    tmag = np.sum(np.abs(dyv * xv * r), axis=0)
    assert np.all(np.abs(orc.decode(dgr, dtype) - dgg) <= uo * np.abs(dgg) + (M + 8) * u32 * tmag)


# --------------------------------------------------------------------------- #
# number formats
# --------------------------------------------------------------------------- #
def test_float16_rounding_matches_numpy():
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 6, 20000),
        [0.0, -0.0, 65504.0, 65519.99, 65520.0, -65520.0, 1e6, 2.0 ** -24, 2.0 ** -25,
         3 * 2.0 ** -26, 2.0 ** -14, 1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, np.inf, -np.inf],
    ])
    ours = orc.encode(vals, "float16")
    with np.errstate(over="ignore"):  # values beyond the float16 range become infinities
        ref = vals.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    back = orc.decode(ours, "float16")
    np.testing.assert_array_equal(back, ref.view(np.float16).astype(np.float64))
    np.testing.assert_array_equal(orc.round_to(vals, "float16"), back)


def test_bfloat16_rounding_matches_torch():
    import torch
    rng = np.random.default_rng(1)
    vals32 = np.concatenate([
        (rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000)).astype(np.float32),
        np.array([0.0, -0.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 3.3895314e38, 3.4e38, 1e-40,
                  np.inf, -np.inf], np.float32),
    ])
    ours = orc.encode(vals32.astype(np.float64), "bfloat16")
    ref = torch.from_numpy(vals32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    # ties to even: 1 + 2^-8 -> 1.0 ; 1 + 3*2^-8 -> 1 + 2^-6
    assert orc.round_to(np.array([1 + 2 ** -8]), "bfloat16")[0] == 1.0
    assert orc.round_to(np.array([1 + 3 * 2 ** -8]), "bfloat16")[0] == 1 + 2 ** -6


def test_float32_rounding_is_c_cast():
    rng = np.random.default_rng(2)
    vals = rng.standard_normal(10000) * 10.0 ** rng.integers(-40, 38, 10000)
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float32)
    np.testing.assert_array_equal(orc.encode(vals, "float32"), ref)
    np.testing.assert_array_equal(orc.decode(ref, "float32"), ref.astype(np.float64))


@pytest.mark.parametrize("dtype", DTYPES)
def test_offset_equals_plain_with_one_plus_w(dtype):
    # With w on a 2^-7 grid in [-1/4, 1/4], 1 + w is exact in every dtype, so the
    # offset variant with w must equal the plain forward/backward with gamma = 1 + w.
    N = 65
    k = np.arange(N) - 32
    w = (k / 128.0).astype(np.float32)
    x = inputs.to_storage(inputs.normal(51, 0, (5, N)), dtype)
    dy = inputs.to_storage(inputs.normal(51, 2, (5, N)), dtype)
    ws, gs = _store(w, dtype), _store(1.0 + w, dtype)
    assert np.array_equal(orc.decode(gs, dtype), 1.0 + orc.decode(ws, dtype))
    yo, ro = orc.fwd_golden(x, ws, dtype, offset=True)
    yp, rp = orc.fwd_golden(x, gs, dtype, offset=False)
    np.testing.assert_allclose(yo, yp, rtol=1e-14)
    np.testing.assert_array_equal(ro, rp)
    dxo, dgo = orc.bwd_golden(dy, x, ws, dtype, offset=True)
    dxp, dgp = orc.bwd_golden(dy, x, gs, dtype, offset=False)
    np.testing.assert_allclose(dxo, dxp, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(dgo, dgp, rtol=1e-14)


# --------------------------------------------------------------------------- #
# the report-only pairwise dgamma reference
# --------------------------------------------------------------------------- #
def _pairwise(t):
    f32 = np.float32
    if len(t) == 0:
        return f32(0)
    if len(t) == 1:
        return t[0]
    mid = len(t) // 2
    return f32(_pairwise(t[:mid]) + _pairwise(t[mid:]))


@pytest.mark.parametrize("dtype", DTYPES)
def test_pairwise_dgamma_reference_brute_force(dtype):
    f32 = np.float32
    M, N = 7, 3
    x, gam, dy = inputs.make_inputs(M, N, dtype, seed=51)
    xv = orc.decode(x, dtype).astype(np.float32)
    dyv = orc.decode(dy, dtype).astype(np.float32)
    _, r = orc.fwd_reference(x, gam, dtype)
    want = np.array([_pairwise([f32(f32(dyv[i, j] * xv[i, j]) * r[i]) for i in range(M)]) for j in range(N)],
                    np.float32)
    np.testing.assert_array_equal(orc.dgamma_pairwise_reference(dy, x, gam, dtype), inputs.to_storage(want, dtype))


def test_pairwise_dgamma_reference_error_bound():
    # pairwise summation: error <= ceil(log2 M) * u32 * sum|terms| (plus the terms' own rounding)
    M, N = 3000, 64
    x, gam, dy = inputs.make_inputs(M, N, "float32", seed=52)
    _, dgg = orc.bwd_golden(dy, x, gam, "float32", want_dx=False)
    pw = orc.dgamma_pairwise_reference(dy, x, gam, "float32").astype(np.float64)
    _, r = orc.fwd_golden(x, gam, "float32")
    mag = np.sum(np.abs(dy.astype(np.float64) * x.astype(np.float64) * r[:, None]), axis=0)
    u32 = 2.0 ** -24
    assert np.all(np.abs(pw - dgg) <= (math.ceil(math.log2(M)) + 4 + N) * u32 * mag)
