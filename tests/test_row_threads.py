"""The threaded row mapper returns exactly what one oracle call returns (CPU)."""
import numpy as np

from oracle import check
from oracle import oracle as orc
from rmsnorm_fwd_bwd_gb300 import inputs

from . import row_threads


def test_chunks_reproduce_one_call_bit_for_bit():
    x, g, dy = inputs.make_inputs(301, 96, "bfloat16", seed=3)
    for threads in (2, 3, 7):
        a = row_threads.map_rows(lambda xx: orc.fwd_golden(xx, g, "bfloat16", eps=1e-6), x,
                                 threads=threads, min_rows=1)
        b = orc.fwd_golden(x, g, "bfloat16", eps=1e-6)
        assert all(np.array_equal(p, q) for p, q in zip(a, b))
        a = row_threads.map_rows(lambda dd, xx: orc.bwd_reference(dd, xx, g, "bfloat16", eps=1e-6)[0], dy, x,
                                 threads=threads, min_rows=1)
        b = orc.bwd_reference(dy, x, g, "bfloat16", eps=1e-6)[0]
        assert np.array_equal(a, b)


def test_gate_with_threads_equals_gate_without():
    x, g, dy = inputs.make_inputs(130, 64, "float32", seed=5)
    yr, rr = orc.fwd_reference(x, g, "float32", eps=1e-6)
    dxr, dgr = orc.bwd_reference(dy, x, g, "float32", eps=1e-6)
    one = check.gate_outputs(x, g, dy, "float32", False, 1e-6, y=yr, rstd=rr, dx=dxr, dgamma=dgr)
    many = check.gate_outputs(x, g, dy, "float32", False, 1e-6, y=yr, rstd=rr, dx=dxr, dgamma=dgr,
                              map_rows=lambda fn, *a: row_threads.map_rows(fn, *a, threads=4, min_rows=1))
    assert [(r.tensor, r.verdict, r.target_error, r.reference_error) for r in one] == \
           [(r.tensor, r.verdict, r.target_error, r.reference_error) for r in many]
