"""The correctness gate accepts the reference and rejects planted mistakes (CPU only).

Mistakes are planted on the CPU, in oracle computations, never in GPU code.
"""
import numpy as np
import pytest

from oracle import gate
from oracle import oracle as orc
from rmsnorm_fwd_bwd_gb300 import inputs


def _case(dtype, M=24, N=257, seed=3, offset=False, x_scale=1.0):
    x, g, dy = inputs.make_inputs(M, N, dtype, seed=seed, offset=offset, x_scale=x_scale)
    yg, rg = orc.fwd_golden(x, g, dtype, offset=offset)
    yr, rr = orc.fwd_reference(x, g, dtype, offset=offset)
    dxg, dgg = orc.bwd_golden(dy, x, g, dtype, offset=offset)
    dxr, dgr = orc.bwd_reference(dy, x, g, dtype, offset=offset)
    return dict(x=x, g=g, dy=dy, yg=yg, rg=rg, yr=orc.decode(yr, dtype), rr=rr.astype(np.float64),
                dxg=dxg, dgg=dgg, dxr=orc.decode(dxr, dtype), dgr=orc.decode(dgr, dtype))


@pytest.mark.parametrize("dtype", ["float32", "float16", "bfloat16"])
def test_reference_passes_its_own_gate(dtype):
    c = _case(dtype)
    rel = gate.FP32_MAX_RELATIVE_ERROR if dtype == "float32" else None
    for name, gold, ref, out in (("y", c["yg"], c["yr"], dtype), ("rstd", c["rg"], c["rr"], "float32"),
                                 ("dx", c["dxg"], c["dxr"], dtype), ("dgamma", c["dgg"], c["dgr"], dtype)):
        res = gate.check(name, gold, ref, ref, out, rel_bound=rel)
        assert res.verdict == "PASS", res.notes


def test_block_denominator_mistake_is_caught():
    # Forward computed as if the masked padding of a 512-wide block counted in the mean.
    dtype = "bfloat16"
    c = _case(dtype, N=257)
    M, N = c["x"].shape
    pad = np.zeros((M, 512), np.uint16)
    pad[:, :N] = c["x"]
    gpad = np.zeros(512, np.uint16)
    gpad[:N] = c["g"]
    yw, _ = orc.fwd_reference(pad, gpad, dtype)
    res = gate.check("y", c["yg"], c["yr"], orc.decode(yw[:, :N], dtype), dtype)
    assert res.verdict == "FAIL"


def test_dgamma_mean_mistake_is_caught():
    dtype = "float32"
    c = _case(dtype, M=17)
    res = gate.check("dgamma", c["dgg"], c["dgr"], c["dgr"] / 17.0, dtype, rel_bound=1e-5)
    assert res.verdict == "FAIL"


def test_dropped_cube_term_is_caught():
    # with x ~ N(0,1) r is close to 1 and r^2 ~ r^3; scale x so that r ~ 1/3
    dtype = "bfloat16"
    c = _case(dtype, x_scale=3.0)
    xv, dyv, gv = (orc.decode(c[k], dtype) for k in ("x", "dy", "g"))
    r = c["rg"][:, None]
    u = dyv * gv
    wrong = orc.round_to(r * u - xv * r * r * np.mean(u * xv, axis=1, keepdims=True), dtype)
    res = gate.check("dx", c["dxg"], c["dxr"], wrong, dtype)
    assert res.verdict == "FAIL"


def test_one_ulp_noise_is_tolerated_but_scaled_noise_is_not():
    dtype = "bfloat16"
    c = _case(dtype)
    gold, ref = c["yg"], c["yr"]
    # a target that rounds the golden correctly passes
    assert gate.check("y", gold, ref, orc.round_to(gold, dtype), dtype).verdict == "PASS"
    # a systematic 1% scale error does not
    assert gate.check("y", gold, ref, orc.round_to(gold * 1.01, dtype), dtype).verdict == "FAIL"


def test_structure_checked_first():
    dtype = "float32"
    c = _case(dtype)
    tgt = c["yr"].copy()
    tgt[3, 5] = np.nan
    res = gate.check("y", c["yg"], c["yr"], tgt, dtype)
    assert res.verdict == "FAIL" and any("NaN" in n for n in res.notes)
    tgt = c["yr"].copy()
    tgt[0, 0] = np.inf
    assert gate.check("y", c["yg"], c["yr"], tgt, dtype).verdict == "FAIL"


def test_inaccurate_reference_makes_gate_invalid():
    dtype = "float32"
    c = _case(dtype)
    bad_ref = c["yg"] * 1.5
    res = gate.check("y", c["yg"], bad_ref, c["yr"], dtype)
    assert res.verdict == "INCONCLUSIVE" and not res.gate_valid
    assert "reference is too inaccurate to gate the target" in res.notes


def test_overflow_to_inf_is_structure_not_error():
    # golden 7e4 does not fit in float16: the output dtype holds +Inf there.
    gold = np.array([1.0, 7e4, -7e4])
    held = orc.round_to(gold, "float16")
    assert np.isposinf(held[1]) and np.isneginf(held[2])
    res = gate.check("y", gold, held, held, "float16")
    assert res.verdict == "PASS"


def test_condition_number():
    assert gate.condition_number([1.0, 2.0, 3.0]) == 1.0
    assert gate.condition_number([1.0, -1.0 + 1e-3]) == pytest.approx((2 - 1e-3) / 1e-3)
    assert gate.condition_number([1.0, -1.0]) == float("inf")


def test_report_table_lists_every_tensor():
    c = _case("bfloat16")
    rs = [gate.check("y", c["yg"], c["yr"], c["yr"], "bfloat16"),
          gate.check("rstd", c["rg"], c["rr"], c["rr"], "float32")]
    text = gate.report("case", rs)
    assert "| y |" in text and "| rstd |" in text and "Overall: PASS" in text


def test_fp32_bound_when_reference_cannot_meet_it():
    # N = 1: dx = r*u*eps/(x^2+eps) cancels; the fp32 reference misses 1e-5 itself.
    x, g, dy = inputs.make_inputs(37, 1, "float32", seed=1)
    dxg, _ = orc.bwd_golden(dy, x, g, "float32")
    dxr, _ = orc.bwd_reference(dy, x, g, "float32")
    dxr = orc.decode(dxr, "float32")
    assert np.max(np.abs(dxr - dxg)) / np.max(np.abs(dxg)) > gate.FP32_MAX_RELATIVE_ERROR
    res = gate.check("dx", dxg, dxr, dxr, "float32", rel_bound=gate.FP32_MAX_RELATIVE_ERROR)
    assert res.verdict == "PASS WITH LIMITATIONS"
    # a target well outside the reference's envelope still fails
    res = gate.check("dx", dxg, dxr, dxg * 1.01, "float32", rel_bound=gate.FP32_MAX_RELATIVE_ERROR)
    assert res.verdict == "FAIL"
    # and on a well-conditioned tensor the bound is enforced
    c = _case("float32")
    res = gate.check("y", c["yg"], c["yr"], c["yg"] * (1 + 3e-5), "float32",
                     rel_bound=gate.FP32_MAX_RELATIVE_ERROR)
    assert res.verdict == "FAIL"
