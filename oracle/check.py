"""Gate a target's RMSNorm outputs against the oracle.

TEST INFRASTRUCTURE: see the package docstring. Takes plain numpy arrays in
storage form (see ``oracle.oracle``); never imports the GPU library.

Every forward output (y, rstd) and every gradient (dx, dgamma) is gated
separately with the same inputs and the same upstream gradient for all three
implementations (page "torchtitan kernel numerics verification", 9-step
workflow, steps 5 and 6).
"""
from __future__ import annotations

import numpy as np

from . import gate
from . import oracle as orc


def _rel_bound(dtype: str):
    return gate.FP32_MAX_RELATIVE_ERROR if dtype == "float32" else None


def _whole(fn, *row_arrays):
    return fn(*row_arrays)


def gate_outputs(x, g, dy, dtype, offset, eps, y=None, rstd=None, dx=None, dgamma=None,
                 rows=None, row_groups=None, map_rows=None):
    """Gate whichever target outputs are given.

    x, g, dy: full inputs (storage form). y, rstd, dx: target outputs for all
    rows, or for ``rows`` only (an index array into the rows of x) when given.
    dgamma: target dgamma over all rows. ``row_groups``: optional {name: row
    indices into the gated rows}; each group is gated on its own as well (a
    stricter check where row classes have very different scales).
    ``map_rows(fn, *row_arrays)``: optional way to evaluate the per-row oracle
    functions (y, rstd, dx), e.g. over row chunks in several threads; it must
    return what ``fn(*row_arrays)`` returns. Every row of those functions is
    computed on its own, so splitting rows does not change a single value.
    Returns a list of ``gate.GateResult``.
    """
    out = []
    xs = x if rows is None else np.ascontiguousarray(x[rows])
    dys = dy if rows is None else np.ascontiguousarray(dy[rows])
    rel = _rel_bound(dtype)
    rowwise = map_rows or _whole
    need_rows = y is not None or rstd is not None or dx is not None
    if need_rows:
        yg, rg = rowwise(lambda xx: orc.fwd_golden(xx, g, dtype, eps=eps, offset=offset, want_y=y is not None), xs)
        yr, rr = rowwise(lambda xx: orc.fwd_reference(xx, g, dtype, eps=eps, offset=offset), xs)
        tensors = []
        if y is not None:
            tensors.append(("y", yg, orc.decode(yr, dtype), orc.decode(y, dtype), dtype))
        if rstd is not None:
            tensors.append(("rstd", rg, rr.astype(np.float64), np.asarray(rstd, np.float64),
                            "float32"))
        if dx is not None:
            dxg = rowwise(lambda dd, xx: orc.bwd_golden(dd, xx, g, dtype, eps=eps, offset=offset)[0], dys, xs)
            dxr = rowwise(lambda dd, xx: orc.bwd_reference(dd, xx, g, dtype, eps=eps, offset=offset)[0], dys, xs)
            tensors.append(("dx", dxg, orc.decode(dxr, dtype), orc.decode(dx, dtype), dtype))
        for name, gold, ref, tgt, odt in tensors:
            out.append(gate.check(name, gold, ref, tgt, odt, rel_bound=rel if name != "rstd" else
                                  gate.FP32_MAX_RELATIVE_ERROR))
            for gname, idx in (row_groups or {}).items():
                idx = np.asarray(idx)
                if idx.size == 0:
                    continue
                out.append(gate.check(f"{name}[{gname}]", gold[idx], ref[idx], tgt[idx], odt,
                                      rel_bound=rel if name != "rstd" else
                                      gate.FP32_MAX_RELATIVE_ERROR))
    if dgamma is not None:
        _, dgg = orc.bwd_golden(dy, x, g, dtype, eps=eps, offset=offset, want_dx=False)
        _, dgr = orc.bwd_reference(dy, x, g, dtype, eps=eps, offset=offset, want_dx=False)
        tgt = orc.decode(dgamma, dtype)
        col = gate.worst_index(dgg, tgt)
        _, rfull = orc.fwd_golden(x, g, dtype, eps=eps, offset=offset, want_y=False)
        cond = None
        if x.shape[0]:
            xc = orc.decode(np.ascontiguousarray(x[:, col]), dtype)
            dyc = orc.decode(np.ascontiguousarray(dy[:, col]), dtype)
            cond = gate.condition_number(dyc * xc * rfull)
        res = gate.check("dgamma", dgg, orc.decode(dgr, dtype), tgt, dtype, rel_bound=rel, condition=cond)
        # report-only: the same terms summed pairwise over rows (a second fp32 reference)
        pw = orc.decode(orc.dgamma_pairwise_reference(dy, x, g, dtype, eps=eps, offset=offset), dtype)
        finite = np.isfinite(dgg)
        if finite.any() and np.isfinite(res.target_error):
            pw_err = float(np.max(np.abs(pw[finite] - dgg[finite])))
            within = res.target_error <= gate.FUDGE_FACTOR * pw_err + res.absolute_floor
            res.notes.append(f"pairwise fp32 reference error {pw_err:.3e} (sequential {res.reference_error:.3e}); "
                             f"target {'within' if within else 'outside'} the gate built on it")
            res.pairwise_error = pw_err
            res.pairwise_within = within
        out.append(res)
    return out


def gate_ln_outputs(x, g, b, dy, dtype, eps, y=None, mean=None, rstd=None, dx=None, dgamma=None,
                    dbeta=None, rows=None):
    """LayerNorm counterpart of ``gate_outputs``: gates whichever of y, mean,
    rstd, dx (all rows, or ``rows`` only), dgamma and dbeta are given.
    Returns a list of ``gate.GateResult``."""
    out = []
    xs = x if rows is None else np.ascontiguousarray(x[rows])
    dys = dy if rows is None else np.ascontiguousarray(dy[rows])
    rel = _rel_bound(dtype)
    fp32 = gate.FP32_MAX_RELATIVE_ERROR
    if y is not None or mean is not None or rstd is not None:
        yg, mg, rg = orc.ln_fwd_golden(xs, g, b, dtype, eps=eps, want_y=y is not None)
        yr, mr, rr = orc.ln_fwd_reference(xs, g, b, dtype, eps=eps)
        if y is not None:
            out.append(gate.check("y", yg, orc.decode(yr, dtype), orc.decode(y, dtype), dtype,
                                  rel_bound=rel))
        if mean is not None:
            out.append(gate.check("mean", mg, mr.astype(np.float64), np.asarray(mean, np.float64),
                                  "float32", rel_bound=fp32))
        if rstd is not None:
            out.append(gate.check("rstd", rg, rr.astype(np.float64), np.asarray(rstd, np.float64),
                                  "float32", rel_bound=fp32))
    if dx is not None:
        dxg, _, _ = orc.ln_bwd_golden(dys, xs, g, dtype, eps=eps)
        dxr, _, _ = orc.ln_bwd_reference(dys, xs, g, dtype, eps=eps)
        out.append(gate.check("dx", dxg, orc.decode(dxr, dtype), orc.decode(dx, dtype), dtype,
                              rel_bound=rel))
    if dgamma is not None or dbeta is not None:
        _, dgg, dbg = orc.ln_bwd_golden(dy, x, g, dtype, eps=eps, want_dx=False)
        _, dgr, dbr = orc.ln_bwd_reference(dy, x, g, dtype, eps=eps, want_dx=False)
        _, mg, rg = orc.ln_fwd_golden(x, g, b, dtype, eps=eps, want_y=False)
        for name, gold, ref, tgt in (("dgamma", dgg, dgr, dgamma), ("dbeta", dbg, dbr, dbeta)):
            if tgt is None:
                continue
            tgt = orc.decode(tgt, dtype)
            cond = None
            if x.shape[0]:
                col = gate.worst_index(gold, tgt)
                dyc = orc.decode(np.ascontiguousarray(dy[:, col]), dtype)
                if name == "dgamma":
                    xc = orc.decode(np.ascontiguousarray(x[:, col]), dtype)
                    cond = gate.condition_number(dyc * (xc - mg) * rg)
                else:
                    cond = gate.condition_number(dyc)
            out.append(gate.check(name, gold, orc.decode(ref, dtype), tgt, dtype, rel_bound=rel,
                                  condition=cond))
    return out


def gate_bwd_bwd_outputs(ddx, ddg, dy, x, g, dtype, offset, eps, d_dy=None, d_x=None, d_gamma=None,
                         rows=None):
    """Gate the RMSNorm double-backward outputs: d_dy and d_x (all rows, or
    ``rows`` only), d_gamma (over all rows). ddg may be None (zero)."""
    out = []
    rel = _rel_bound(dtype)
    if d_dy is not None or d_x is not None:
        sl = (lambda a: a) if rows is None else (lambda a: np.ascontiguousarray(a[rows]))
        G = orc.bwd_bwd_golden(sl(ddx), ddg, sl(dy), sl(x), g, dtype, eps=eps, offset=offset)
        R = orc.bwd_bwd_reference(sl(ddx), ddg, sl(dy), sl(x), g, dtype, eps=eps, offset=offset)
        for name, gold, ref, tgt in (("d_dy", G[0], R[0], d_dy), ("d_x", G[1], R[1], d_x)):
            if tgt is not None:
                out.append(gate.check(name, gold, orc.decode(ref, dtype), orc.decode(tgt, dtype), dtype,
                                      rel_bound=rel))
    if d_gamma is not None:
        G = orc.bwd_bwd_golden(ddx, ddg, dy, x, g, dtype, eps=eps, offset=offset)
        R = orc.bwd_bwd_reference(ddx, ddg, dy, x, g, dtype, eps=eps, offset=offset)
        out.append(gate.check("d_gamma", G[2], orc.decode(R[2], dtype), orc.decode(d_gamma, dtype), dtype,
                              rel_bound=rel))
    return out
