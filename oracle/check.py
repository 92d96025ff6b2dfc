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


def gate_outputs(x, g, dy, dtype, offset, eps, y=None, rstd=None, dx=None, dgamma=None,
                 rows=None, row_groups=None):
    """Gate whichever target outputs are given.

    x, g, dy: full inputs (storage form). y, rstd, dx: target outputs for all
    rows, or for ``rows`` only (an index array into the rows of x) when given.
    dgamma: target dgamma over all rows. ``row_groups``: optional {name: row
    indices into the gated rows}; each group is gated on its own as well (a
    stricter check where row classes have very different scales).
    Returns a list of ``gate.GateResult``.
    """
    out = []
    xs = x if rows is None else np.ascontiguousarray(x[rows])
    dys = dy if rows is None else np.ascontiguousarray(dy[rows])
    rel = _rel_bound(dtype)
    need_rows = y is not None or rstd is not None or dx is not None
    if need_rows:
        yg, rg = orc.fwd_golden(xs, g, dtype, eps=eps, offset=offset, want_y=y is not None)
        yr, rr = orc.fwd_reference(xs, g, dtype, eps=eps, offset=offset)
        tensors = []
        if y is not None:
            tensors.append(("y", yg, orc.decode(yr, dtype), orc.decode(y, dtype), dtype))
        if rstd is not None:
            tensors.append(("rstd", rg, rr.astype(np.float64), np.asarray(rstd, np.float64),
                            "float32"))
        if dx is not None:
            dxg, _ = orc.bwd_golden(dys, xs, g, dtype, eps=eps, offset=offset)
            dxr, _ = orc.bwd_reference(dys, xs, g, dtype, eps=eps, offset=offset)
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
        out.append(gate.check("dgamma", dgg, orc.decode(dgr, dtype), tgt, dtype, rel_bound=rel,
                              condition=cond))
    return out
