"""Pins of the RMSNorm double-backward oracle (CPU only).

The double backward is the gradient of L = sum(ddx * dx) + sum(ddg * dgamma)
with respect to the backward's inputs dy, x and gamma (the page "Check an AI
model calculation before accelerating it", section "Adapting the kernel and
moving to production", lists double backward among the unvalidated
extensions). The golden closed form is pinned against central finite
differences of the golden backward -- itself pinned by finite differences of
the forward and by the pages' worked examples -- plus linearity and zero cases;
the fp32 reference against a scalar float32 loop and an error bound.
"""
import numpy as np
import pytest

from oracle import oracle as orc
from rmsnorm_fwd_bwd_gb300 import inputs

DTYPES = ["float32", "float16", "bfloat16"]


def _grid(a, q=2.0 ** -8):
    return (np.round(np.asarray(a, np.float64) / q) * q).astype(np.float32)


@pytest.mark.parametrize("offset", [False, True])
def test_finite_differences_of_the_backward(offset):
    M, N = 3, 6
    x = _grid(inputs.normal(31, 0, (M, N)))
    dy = _grid(inputs.normal(31, 2, (M, N)))
    g = _grid((0.0 if offset else 1.0) + inputs.normal(31, 1, (N,), 0.3))
    ddx = inputs.normal(31, 3, (M, N))
    ddg = inputs.normal(31, 4, (N,))
    eps = 1e-2
    ddxd, ddgd = ddx.astype(np.float64), ddg.astype(np.float64)
    h = 2.0 ** -12

    def L(dya, xa, ga):
        dx, dg = orc.bwd_golden(dya, xa, ga, "float32", eps=eps, offset=offset)
        return float(np.sum(ddxd * dx) + np.sum(ddgd * dg))

    def fd(arr, idx, f):
        p = arr.copy(); p[idx] += np.float32(h)
        m = arr.copy(); m[idx] -= np.float32(h)
        return (f(p) - f(m)) / (2 * h)

    d_dy, d_x, d_g = orc.bwd_bwd_golden(ddx, ddg, dy, x, g, "float32", eps=eps, offset=offset)
    fd_dy = np.array([[fd(dy, (i, j), lambda a: L(a, x, g)) for j in range(N)] for i in range(M)])
    fd_x = np.array([[fd(x, (i, j), lambda a: L(dy, a, g)) for j in range(N)] for i in range(M)])
    fd_g = np.array([fd(g, j, lambda a: L(dy, x, a)) for j in range(N)])
    np.testing.assert_allclose(d_dy, fd_dy, atol=1e-6 * np.max(np.abs(d_dy)), rtol=0)
    np.testing.assert_allclose(d_x, fd_x, atol=1e-5 * np.max(np.abs(d_x)), rtol=0)
    np.testing.assert_allclose(d_g, fd_g, atol=1e-6 * np.max(np.abs(d_g)), rtol=0)


def test_linear_in_the_cotangents_and_zero_for_zero():
    M, N = 4, 33
    x, g, dy = inputs.make_inputs(M, N, "float32", seed=32)
    ddx = inputs.normal(32, 3, (M, N))
    ddg = inputs.normal(32, 4, (N,))
    zero_x = np.zeros((M, N), np.float32)
    full = orc.bwd_bwd_golden(ddx, ddg, dy, x, g, "float32")
    only_x = orc.bwd_bwd_golden(ddx, None, dy, x, g, "float32")
    only_g = orc.bwd_bwd_golden(zero_x, ddg, dy, x, g, "float32")
    for a, b, c in zip(full, only_x, only_g):
        np.testing.assert_allclose(a, b + c, rtol=1e-13, atol=1e-13 * np.max(np.abs(a)))
    for a in orc.bwd_bwd_golden(zero_x, None, dy, x, g, "float32"):
        assert np.all(a == 0)
    # ddg alone: d_dy = r * x * ddg and d_gamma = 0 (dgamma does not depend on gamma)
    _, r = orc.fwd_golden(x, g, "float32")
    np.testing.assert_allclose(only_g[0], r[:, None] * x.astype(np.float64) * ddg.astype(np.float64),
                               rtol=1e-14, atol=0)
    assert np.all(only_g[2] == 0)


def test_single_column_closed_form():
    # N = 1: dx = eps * g * dy * r^3, so d_dy = eps * g * r^3 * ddx (ddg = 0)
    x = np.array([[0.5], [-2.0], [3.0]], np.float32)
    dy = np.array([[1.0], [0.25], [-1.5]], np.float32)
    g = np.array([1.25], np.float32)
    ddx = np.array([[2.0], [-1.0], [0.5]], np.float32)
    eps = 0.125
    d_dy, _, _ = orc.bwd_bwd_golden(ddx, None, dy, x, g, "float32", eps=eps)
    r = 1.0 / np.sqrt(x.astype(np.float64) ** 2 + eps)
    np.testing.assert_allclose(d_dy, eps * 1.25 * r ** 3 * ddx, rtol=1e-14)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("offset", [False, True])
def test_reference_brute_force(dtype, offset):
    M, N = 3, 7
    f32 = np.float32
    x, gam, dy = inputs.make_inputs(M, N, dtype, seed=43, offset=offset)
    ddx = inputs.to_storage(inputs.normal(43, 3, (M, N)), dtype)
    ddg = inputs.to_storage(inputs.normal(43, 4, (N,)), dtype)
    xv, gv, dyv, tv, qv = (orc.decode(a, dtype).astype(np.float32) for a in (x, gam, dy, ddx, ddg))
    eps = f32(1e-6)
    o_dy = np.zeros((M, N), np.float32)
    o_x = np.zeros((M, N), np.float32)
    acc = [f32(0)] * N
    with np.errstate(all="ignore"):
        for i in range(M):
            ss = f32(0)
            for j in range(N):
                ss = f32(ss + f32(xv[i, j] * xv[i, j]))
            r = f32(f32(1) / f32(np.sqrt(f32(f32(ss / f32(N)) + eps))))
            sc = sa = sb = sd = f32(0)
            for j in range(N):
                g = f32(f32(1) + gv[j]) if offset else gv[j]
                u = f32(dyv[i, j] * g)
                sc = f32(sc + f32(u * xv[i, j]))
                sa = f32(sa + f32(tv[i, j] * xv[i, j]))
                sb = f32(sb + f32(tv[i, j] * u))
                sd = f32(sd + f32(f32(qv[j] * dyv[i, j]) * xv[i, j]))
            c, A, Bm, D = (f32(v / f32(N)) for v in (sc, sa, sb, sd))
            r2 = f32(r * r)
            r3 = f32(r2 * r)
            r5 = f32(r3 * r2)
            k5 = f32(f32(f32(3) * r5) * f32(c * A))
            bd = f32(Bm + D)
            for j in range(N):
                g = f32(f32(1) + gv[j]) if offset else gv[j]
                u = f32(dyv[i, j] * g)
                e = f32(tv[i, j] - f32(f32(r2 * xv[i, j]) * A))
                o_dy[i, j] = f32(f32(f32(g * r) * e) + f32(f32(r * xv[i, j]) * qv[j]))
                inner = f32(f32(f32(c * tv[i, j]) + f32(u * A)) + f32(xv[i, j] * bd))
                o_x[i, j] = f32(f32(f32(f32(r * qv[j]) * dyv[i, j]) - f32(r3 * inner)) + f32(k5 * xv[i, j]))
                acc[j] = f32(acc[j] + f32(f32(r * dyv[i, j]) * e))
    d_dy, d_x, d_g = orc.bwd_bwd_reference(ddx, ddg, dy, x, gam, dtype, offset=offset)
    np.testing.assert_array_equal(d_dy, inputs.to_storage(o_dy, dtype))
    np.testing.assert_array_equal(d_x, inputs.to_storage(o_x, dtype))
    np.testing.assert_array_equal(d_g, inputs.to_storage(np.array(acc, np.float32), dtype))


@pytest.mark.parametrize("dtype", DTYPES)
def test_reference_close_to_golden(dtype):
    # fp32 error analysis: each output within its own rounding plus a small
    # multiple of u32 times the magnitudes of the terms it is built from (sums
    # of N terms for the row statistics, of M terms for d_gamma).
    M, N = 16, 512
    x, g, dy = inputs.make_inputs(M, N, dtype, seed=9)
    ddx = inputs.to_storage(inputs.normal(9, 3, (M, N)), dtype)
    ddg = inputs.to_storage(inputs.normal(9, 4, (N,)), dtype)
    G = orc.bwd_bwd_golden(ddx, ddg, dy, x, g, dtype)
    R = [orc.decode(a, dtype) for a in orc.bwd_bwd_reference(ddx, ddg, dy, x, g, dtype)]
    u32 = 2.0 ** -24
    uo = {"float32": 2.0 ** -24, "float16": 2.0 ** -11, "bfloat16": 2.0 ** -8}[dtype]
    xv, gv, dyv, tv, qv = (orc.decode(a, dtype) for a in (x, g, dy, ddx, ddg))
    _, r = orc.fwd_golden(x, g, dtype)
    r = r[:, None]
    u = dyv * gv
    mA = np.mean(np.abs(tv * xv), axis=1, keepdims=True)
    mB = np.mean(np.abs(tv * u), axis=1, keepdims=True)
    mC = np.mean(np.abs(u * xv), axis=1, keepdims=True)
    mD = np.mean(np.abs(qv * dyv * xv), axis=1, keepdims=True)
    k = (N + 32) * u32
    mag_dy = np.abs(gv) * r * (np.abs(tv) + r ** 2 * np.abs(xv) * mA) + r * np.abs(xv * qv)
    mag_x = (r * np.abs(qv * dyv) + r ** 3 * (mC * np.abs(tv) + np.abs(u) * mA + np.abs(xv) * (mB + mD))
             + 3 * r ** 5 * mC * mA * np.abs(xv))
    assert np.all(np.abs(R[0] - G[0]) <= uo * np.abs(G[0]) + k * mag_dy + 1e-30)
    assert np.all(np.abs(R[1] - G[1]) <= uo * np.abs(G[1]) + k * mag_x + 1e-30)
    tg = np.sum(r * np.abs(dyv) * (np.abs(tv) + r ** 2 * np.abs(xv) * mA), axis=0)
    assert np.all(np.abs(R[2] - G[2]) <= uo * np.abs(G[2]) + (M + N + 32) * u32 * tg + 1e-30)


@pytest.mark.parametrize("dtype", DTYPES)
def test_gate_accepts_reference_and_rejects_a_dropped_term(dtype):
    from oracle import check, gate
    M, N = 24, 200
    x, g, dy = inputs.make_inputs(M, N, dtype, seed=10)
    ddx = inputs.to_storage(inputs.normal(10, 3, (M, N)), dtype)
    ddg = inputs.to_storage(inputs.normal(10, 4, (N,)), dtype)
    R = orc.bwd_bwd_reference(ddx, ddg, dy, x, g, dtype)
    res = check.gate_bwd_bwd_outputs(ddx, ddg, dy, x, g, dtype, False, 1e-6, d_dy=R[0], d_x=R[1], d_gamma=R[2])
    assert gate.overall(res) == "PASS", gate.report("reference as target", res)
    # a target that drops the r*x*ddg term of d_dy
    G = orc.bwd_bwd_golden(ddx, ddg, dy, x, g, dtype)
    _, r = orc.fwd_golden(x, g, dtype)
    bad = orc.encode(G[0] - r[:, None] * orc.decode(x, dtype) * orc.decode(ddg, dtype), dtype)
    assert gate.overall(check.gate_bwd_bwd_outputs(ddx, ddg, dy, x, g, dtype, False, 1e-6, d_dy=bad)) == "FAIL"
