"""Pins of the LayerNorm oracle to facts outside itself (CPU only).

The LayerNorm page ("torch.compile performance leap: optimizing LayerNorm and
RMSNorm kernels", sections 1.1 and 2) names the operation -- per-row mean and
variance, learned gamma and beta, and gradients for the input, the weight and
the bias -- but prints no numbers. So these pins are closed forms worked by
hand, invariants of the definition, finite differences of the forward, and
brute force on tiny inputs.
"""
import math

import numpy as np
import pytest

from oracle import oracle as orc
from rmsnorm_fwd_bwd_gb300 import inputs

DTYPES = ["float32", "float16", "bfloat16"]


def _f32(v):
    return np.asarray(v, np.float32)


# --------------------------------------------------------------------------- #
# hand-worked closed forms
# --------------------------------------------------------------------------- #
def test_four_element_row_by_hand():
    # x = 1, 2, 3, 4: mean 5/2, variance (9 + 1 + 1 + 9)/16 = 5/4, so with eps = 0
    # x_hat = (-3, -1, 1, 3) / sqrt(5) and r = 2 / sqrt(5).
    x = _f32([[1, 2, 3, 4]])
    g = _f32([1.0, 2.0, 0.5, -1.0])
    b = _f32([0.5, 0.0, -1.0, 2.0])
    y, mean, rstd = orc.ln_fwd_golden(x, g, b, "float32", eps=0.0)
    s5 = math.sqrt(5.0)
    xh = np.array([-3, -1, 1, 3]) / s5
    assert mean[0] == 2.5
    assert abs(rstd[0] - 2 / s5) < 1e-15
    np.testing.assert_allclose(y[0], xh * g + b, rtol=0, atol=1e-15)
    # dy = e_0, gamma = 1: u = e_0, mean(u) = 1/4, mean(u x_hat) = -3/(4 sqrt 5);
    # dx_j = r (u_j - 1/4 + x_hat_j * 3/(4 sqrt 5))
    dy = _f32([[1, 0, 0, 0]])
    dx, dg, db = orc.ln_bwd_golden(dy, x, np.ones(4, np.float32), "float32", eps=0.0)
    want = (2 / s5) * (np.array([1, 0, 0, 0]) - 0.25 + xh * 3 / (4 * s5))
    np.testing.assert_allclose(dx[0], want, rtol=0, atol=1e-15)
    np.testing.assert_allclose(dx[0], [0.3 * 2 / s5, -0.4 * 2 / s5, -0.1 * 2 / s5, 0.2 * 2 / s5],
                               rtol=0, atol=1e-15)
    np.testing.assert_allclose(dg, [-3 / s5, 0, 0, 0], rtol=0, atol=1e-15)
    np.testing.assert_array_equal(db, [1, 0, 0, 0])


@pytest.mark.parametrize("dtype", DTYPES)
def test_two_columns_have_no_input_gradient(dtype):
    # N = 2, eps = 0: x_hat = (-1, +1) whatever x is (if x_0 < x_1), so y does not
    # depend on x and dx = 0 exactly in the golden arithmetic up to rounding.
    x = inputs.to_storage(_f32([[0.5, 3.0], [-7.0, 2.0], [1.0, 1.25]]), dtype)
    g = inputs.to_storage(_f32([1.5, -0.75]), dtype)
    b = inputs.to_storage(_f32([0.25, 0.5]), dtype)
    dy = inputs.to_storage(_f32([[1.0, -2.0], [0.3, 0.9], [-4.0, 4.0]]), dtype)
    y, _, _ = orc.ln_fwd_golden(x, g, b, dtype, eps=0.0)
    gv, bv = orc.decode(g, dtype), orc.decode(b, dtype)
    np.testing.assert_allclose(y, np.tile([-gv[0] + bv[0], gv[1] + bv[1]], (3, 1)), atol=1e-15)
    dx, dg, db = orc.ln_bwd_golden(dy, x, g, dtype, eps=0.0)
    assert np.max(np.abs(dx)) < 1e-14
    dyv = orc.decode(dy, dtype)
    np.testing.assert_allclose(dg, [-np.sum(dyv[:, 0]), np.sum(dyv[:, 1])], atol=1e-14)
    np.testing.assert_allclose(db, np.sum(dyv, axis=0), atol=1e-14)


@pytest.mark.parametrize("dtype", DTYPES)
def test_constant_rows(dtype):
    # A constant row has variance 0: x_hat = 0, y = beta, r = 1/sqrt(eps), and
    # dx = r * (u - mean(u)).
    eps = 0.0625
    x = inputs.to_storage(np.full((2, 6), 3.5, np.float32), dtype)
    g = inputs.to_storage(_f32([1, 2, 3, -1, 0.5, 0.25]), dtype)
    b = inputs.to_storage(_f32([0.1, -0.2, 0.3, 0, 1, 2]), dtype)
    dy = inputs.to_storage(_f32([[1, 0, 2, 0, -1, 4], [0, 0, 0, 0, 0, 1]]), dtype)
    y, mean, rstd = orc.ln_fwd_golden(x, g, b, dtype, eps=eps)
    np.testing.assert_array_equal(y, np.tile(orc.decode(b, dtype), (2, 1)))
    np.testing.assert_array_equal(mean, [3.5, 3.5])
    np.testing.assert_array_equal(rstd, [4.0, 4.0])
    dx, dg, _ = orc.ln_bwd_golden(dy, x, g, dtype, eps=eps)
    u = orc.decode(dy, dtype) * orc.decode(g, dtype)
    np.testing.assert_allclose(dx, 4.0 * (u - u.mean(axis=1, keepdims=True)), atol=1e-14)
    np.testing.assert_array_equal(dg, np.zeros(6))
    # the fp32 reference reaches the same exact values
    yr, mr, rr = orc.ln_fwd_reference(x, g, b, dtype, eps=eps)
    np.testing.assert_array_equal(yr, np.tile(b, (2, 1)))
    np.testing.assert_array_equal(rr, [4.0, 4.0])


def test_single_column():
    # N = 1: mean = x, variance 0, y = beta, dx = r * (u - u) = 0, dgamma = 0, dbeta = sum dy.
    x = _f32([[2.0], [-5.0], [0.0]])
    dy = _f32([[1.0], [2.0], [-0.5]])
    g, b = _f32([3.0]), _f32([-1.0])
    y, mean, rstd = orc.ln_fwd_golden(x, g, b, "float32", eps=0.25)
    np.testing.assert_array_equal(y, [[-1.0]] * 3)
    np.testing.assert_array_equal(mean, [2, -5, 0])
    np.testing.assert_array_equal(rstd, [2, 2, 2])
    dx, dg, db = orc.ln_bwd_golden(dy, x, g, "float32", eps=0.25)
    np.testing.assert_array_equal(dx, np.zeros((3, 1)))
    np.testing.assert_array_equal(dg, [0.0])
    np.testing.assert_array_equal(db, [2.5])


# --------------------------------------------------------------------------- #
# invariants of the definition
# --------------------------------------------------------------------------- #
def test_shift_and_scale_invariance():
    # y(x + c) = y(x) and, with eps = 0, y(2^k x) = y(x); integer-valued x keeps
    # the shifted and scaled inputs exact in float32.
    rng = np.random.default_rng(3)
    x = rng.integers(-50, 50, (5, 33)).astype(np.float32)
    x[:, 0] += 1  # no constant rows
    g = _f32(1 + 0.1 * rng.standard_normal(33))
    b = _f32(0.1 * rng.standard_normal(33))
    y0, m0, r0 = orc.ln_fwd_golden(x, g, b, "float32", eps=0.0)
    y1, m1, r1 = orc.ln_fwd_golden(x + np.float32(4096), g, b, "float32", eps=0.0)
    y2, _, r2 = orc.ln_fwd_golden(x * np.float32(8), g, b, "float32", eps=0.0)
    np.testing.assert_allclose(y1, y0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(m1, m0 + 4096, rtol=1e-15)
    np.testing.assert_allclose(r1, r0, rtol=1e-13)
    np.testing.assert_allclose(y2, y0, rtol=0, atol=1e-13)
    np.testing.assert_allclose(r2, r0 / 8, rtol=1e-14)


def test_zero_mean_rows_match_rmsnorm():
    # Rows made of +a, -a pairs have mean exactly 0; LayerNorm then equals
    # RMSNorm (variance = mean of squares) plus beta.
    rng = np.random.default_rng(4)
    half = _f32(rng.standard_normal((6, 20)))
    x = np.concatenate([half, -half], axis=1)
    g = _f32(1 + 0.1 * rng.standard_normal(40))
    b = _f32(0.1 * rng.standard_normal(40))
    y, mean, rstd = orc.ln_fwd_golden(x, g, b, "float32", eps=1e-6)
    y_rms, r_rms = orc.fwd_golden(x, g, "float32", eps=1e-6)
    assert np.max(np.abs(mean)) < 1e-15
    np.testing.assert_allclose(rstd, r_rms, rtol=1e-14)
    np.testing.assert_allclose(y, y_rms + b.astype(np.float64), rtol=0, atol=1e-13)


def test_input_gradient_rows_sum_to_zero():
    # sum_j dx_j = r * (sum u - N mean(u) - mean(u x_hat) sum x_hat) = 0 because
    # sum x_hat = 0, for any gamma and eps.
    x, g, b, dy = inputs.make_ln_inputs(7, 90, "float32", seed=5)
    dx, _, _ = orc.ln_bwd_golden(dy, x, g, "float32", eps=0.5)
    scale = np.max(np.abs(dx))
    assert np.max(np.abs(dx.sum(axis=1))) < 1e-13 * 90 * scale


def test_bias_gradient_is_column_sums_of_dy():
    x, g, b, dy = inputs.make_ln_inputs(33, 17, "bfloat16", seed=6)
    _, _, db = orc.ln_bwd_golden(dy, x, g, "bfloat16")
    dyv = orc.decode(dy, "bfloat16")
    for j in range(17):
        assert abs(db[j] - math.fsum(dyv[:, j])) <= 1e-13 * math.fsum(np.abs(dyv[:, j]))


# --------------------------------------------------------------------------- #
# finite differences of the golden forward
# --------------------------------------------------------------------------- #
def test_backward_finite_differences():
    """Central differences of L = sum(dy * y) against the golden dx, dgamma and
    dbeta. Inputs on a 2^-8 grid so that +/- 2^-12 steps are exact in float32."""
    M, N = 3, 6
    q = 2.0 ** -8
    x = (np.round((inputs.normal(22, 0, (M, N)) + inputs.normal(22, 5, (M, 1), 2.0)) / q) * q).astype(np.float32)
    g = (np.round((np.float32(1) + inputs.normal(22, 1, (N,), 0.3)) / q) * q).astype(np.float32)
    b = (np.round(inputs.normal(22, 6, (N,), 0.3) / q) * q).astype(np.float32)
    dy = inputs.normal(22, 2, (M, N))
    dyd = dy.astype(np.float64)
    h = 2.0 ** -12
    eps = 1e-2

    def loss(xa, ga, ba):
        y, _, _ = orc.ln_fwd_golden(xa, ga, ba, "float32", eps=eps)
        return float(np.sum(dyd * y))

    dx, dg, db = orc.ln_bwd_golden(dy, x, g, "float32", eps=eps)

    def fd(arr, idx, f):
        p = arr.copy(); p[idx] += np.float32(h)
        m = arr.copy(); m[idx] -= np.float32(h)
        return (f(p) - f(m)) / (2 * h)

    fd_x = np.array([[fd(x, (i, j), lambda a: loss(a, g, b)) for j in range(N)] for i in range(M)])
    fd_g = np.array([fd(g, j, lambda a: loss(x, a, b)) for j in range(N)])
    fd_b = np.array([fd(b, j, lambda a: loss(x, g, a)) for j in range(N)])
    np.testing.assert_allclose(dx, fd_x, atol=2e-6 * np.max(np.abs(dx)), rtol=0)
    np.testing.assert_allclose(dg, fd_g, atol=2e-6 * np.max(np.abs(dg)), rtol=0)
    np.testing.assert_allclose(db, fd_b, atol=1e-9, rtol=0)


# --------------------------------------------------------------------------- #
# reference (fp32 intermediates): brute force and error bounds
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("dtype", DTYPES)
def test_reference_brute_force(dtype):
    """Tiny inputs: an independent scalar-by-scalar float32 loop (numpy scalars)."""
    M, N = 3, 7
    f32 = np.float32
    x, g, b, dy = inputs.make_ln_inputs(M, N, dtype, seed=42, x_scale=1.3)
    xv = orc.decode(x, dtype).astype(np.float32)
    gv = orc.decode(g, dtype).astype(np.float32)
    bv = orc.decode(b, dtype).astype(np.float32)
    dyv = orc.decode(dy, dtype).astype(np.float32)
    eps = f32(1e-5)
    y_bf = np.zeros((M, N), np.float32)
    dx_bf = np.zeros((M, N), np.float32)
    m_bf = np.zeros(M, np.float32)
    r_bf = np.zeros(M, np.float32)
    accg = [f32(0)] * N
    accb = [f32(0)] * N
    with np.errstate(all="ignore"):
        for i in range(M):
            s = f32(0)
            for j in range(N):
                s = f32(s + xv[i, j])
            mu = f32(s / f32(N))
            v = f32(0)
            for j in range(N):
                d = f32(xv[i, j] - mu)
                v = f32(v + f32(d * d))
            r = f32(f32(1) / f32(np.sqrt(f32(f32(v / f32(N)) + eps))))
            m_bf[i], r_bf[i] = mu, r
            su = f32(0)
            suh = f32(0)
            for j in range(N):
                u = f32(dyv[i, j] * gv[j])
                xh = f32(f32(xv[i, j] - mu) * r)
                su = f32(su + u)
                suh = f32(suh + f32(u * xh))
            a1 = f32(su / f32(N))
            a2 = f32(suh / f32(N))
            for j in range(N):
                xh = f32(f32(xv[i, j] - mu) * r)
                y_bf[i, j] = f32(f32(xh * gv[j]) + bv[j])
                u = f32(dyv[i, j] * gv[j])
                dx_bf[i, j] = f32(r * f32(f32(u - a1) - f32(xh * a2)))
                accg[j] = f32(accg[j] + f32(dyv[i, j] * xh))
                accb[j] = f32(accb[j] + dyv[i, j])
    y, mean, rstd = orc.ln_fwd_reference(x, g, b, dtype)
    dx, dg, db = orc.ln_bwd_reference(dy, x, g, dtype)
    np.testing.assert_array_equal(mean, m_bf)
    np.testing.assert_array_equal(rstd, r_bf)
    np.testing.assert_array_equal(y, inputs.to_storage(y_bf, dtype))
    np.testing.assert_array_equal(dx, inputs.to_storage(dx_bf, dtype))
    np.testing.assert_array_equal(dg, inputs.to_storage(np.array(accg, np.float32), dtype))
    np.testing.assert_array_equal(db, inputs.to_storage(np.array(accb, np.float32), dtype))


@pytest.mark.parametrize("dtype", DTYPES)
def test_reference_close_to_golden(dtype):
    # fp32 error analysis: the mean is within N u32 |x|max of its value, the
    # variance (two-pass) within a few N u32 of it relatively, and each output
    # within its own rounding plus a small multiple of u32 times the magnitudes
    # it is built from.
    M, N = 16, 512
    x, g, b, dy = inputs.make_ln_inputs(M, N, dtype, seed=8)
    yg, mg, rg = orc.ln_fwd_golden(x, g, b, dtype)
    yr, mr, rr = orc.ln_fwd_reference(x, g, b, dtype)
    u32 = 2.0 ** -24
    uo = {"float32": 2.0 ** -24, "float16": 2.0 ** -11, "bfloat16": 2.0 ** -8}[dtype]
    xv, gv, bv, dyv = (orc.decode(a, dtype) for a in (x, g, b, dy))
    amax = np.max(np.abs(xv), axis=1)
    assert np.all(np.abs(mr - mg) <= (N + 4) * u32 * amax)
    assert np.all(np.abs(rr - rg) <= (2 * N + 16) * u32 * rg * (1 + amax * rg))
    xh = (xv - mg[:, None]) * rg[:, None]
    # y picks up the mean's error times r and the relative error of r times x_hat
    stat = (2 * N + 16) * u32 * (1 + amax[:, None] * rg[:, None]) * (1 + np.abs(xh)) * np.abs(gv)
    bound_y = uo * np.abs(yg) + 4 * u32 * (np.abs(xh * gv) + np.abs(bv)) + stat
    assert np.all(np.abs(orc.decode(yr, dtype) - yg) <= bound_y + 1e-30)
    dxg, dgg, dbg = orc.ln_bwd_golden(dy, x, g, dtype)
    dxr, dgr, dbr = orc.ln_bwd_reference(dy, x, g, dtype)
    u = dyv * gv
    k = (1 + amax[:, None] * rg[:, None])
    mag = rg[:, None] * (np.abs(u) + np.mean(np.abs(u), axis=1, keepdims=True)
                         + np.abs(xh) * np.mean(np.abs(u * xh), axis=1, keepdims=True))
    bound = uo * np.abs(dxg) + (N + 16) * u32 * k * mag
    assert np.all(np.abs(orc.decode(dxr, dtype) - dxg) <= bound + 1e-30)
    tg = np.sum(np.abs(dyv * xh) * k, axis=0)
    assert np.all(np.abs(orc.decode(dgr, dtype) - dgg) <= uo * np.abs(dgg) + (M + 2 * N + 16) * u32 * tg)
    tb = np.sum(np.abs(dyv), axis=0)
    assert np.all(np.abs(orc.decode(dbr, dtype) - dbg) <= uo * np.abs(dbg) + (M + 2) * u32 * tb)


# --------------------------------------------------------------------------- #
# the gate on LayerNorm outputs
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("dtype", DTYPES)
def test_gate_accepts_reference_and_rejects_a_dropped_term(dtype):
    from oracle import check, gate
    M, N = 24, 200
    x, g, b, dy = inputs.make_ln_inputs(M, N, dtype, seed=9)
    y, mean, rstd = orc.ln_fwd_reference(x, g, b, dtype)
    dx, dg, db = orc.ln_bwd_reference(dy, x, g, dtype)
    res = check.gate_ln_outputs(x, g, b, dy, dtype, 1e-5, y=y, mean=mean, rstd=rstd, dx=dx,
                                dgamma=dg, dbeta=db)
    assert gate.overall(res) == "PASS", gate.report("reference as target", res)
    # a target that forgets the mean(u) term of dx
    dxg, _, _ = orc.ln_bwd_golden(dy, x, g, dtype)
    u = orc.decode(dy, dtype) * orc.decode(g, dtype)
    bad = orc.encode(dxg + rstd[:, None].astype(np.float64) * u.mean(axis=1, keepdims=True), dtype)
    res = check.gate_ln_outputs(x, g, b, dy, dtype, 1e-5, dx=bad)
    assert gate.overall(res) == "FAIL"
    # a target whose mean is off by 2^-10 relative
    res = check.gate_ln_outputs(x, g, b, dy, dtype, 1e-5,
                                mean=(mean.astype(np.float64) * (1 + 2.0 ** -10)).astype(np.float32))
    assert gate.overall(res) == "FAIL"
