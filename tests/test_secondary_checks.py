"""The pages' secondary closeness check and the reduction growth analysis,
pinned on the CPU (no GPU): tolerances and worked numbers as printed, planted
mistakes caught, synthetic growth laws classified as the page describes."""
import numpy as np
import pytest

from oracle import gate, growth
from oracle import oracle as orc
from rmsnorm_fwd_bwd_gb300 import inputs


# --------------------------------------------------------------------------- #
# closeness check
# --------------------------------------------------------------------------- #
def test_declared_tolerances_are_the_pages(golden_file):
    f = golden_file("allclose_tolerances.txt")
    assert gate.ALLCLOSE_TOLERANCES["float32"] == (f["fp32_atol"][0][0], f["fp32_rtol"][0][0])
    assert gate.ALLCLOSE_TOLERANCES["float16"] == (f["fp16_atol"][0][0], f["fp16_rtol"][0][0])
    assert "bfloat16" not in gate.ALLCLOSE_TOLERANCES  # the page declares none


def test_printed_examples_of_the_rule(golden_file):
    f = golden_file("allclose_tolerances.txt")
    refs, allowed = f["example_reference"][0], f["example_allowed"][0]
    for r, a in zip(refs, allowed):
        assert gate.allowed_difference(r, "float32") == pytest.approx(a, rel=1e-12)


@pytest.mark.parametrize("dtype", ["float32", "float16"])
def test_reference_is_close_to_itself_and_a_planted_mistake_is_not(dtype):
    x, g, dy = inputs.make_inputs(40, 96, dtype, seed=2)
    _, dgr = orc.bwd_reference(dy, x, g, dtype)
    ref = orc.decode(dgr, dtype)
    assert gate.allclose("dgamma", ref, ref, dtype).passed
    wrong = ref / x.shape[0]  # dgamma as a mean over rows
    res = gate.allclose("dgamma", wrong, ref, dtype)
    assert not res.passed and res.failing > 0 and res.worst_excess > 0


def test_one_element_over_the_tolerance_fails():
    ref = np.array([1.0, 100.0, -3.0, 0.0])
    allowed = gate.allowed_difference(ref, "float32")
    inside = ref + 0.999 * allowed
    assert gate.allclose("t", inside, ref, "float32").passed
    outside = inside.copy()
    outside[1] = ref[1] + 1.001 * allowed[1]
    res = gate.allclose("t", outside, ref, "float32")
    assert res.failing == 1 and res.worst_excess > 0


def test_special_values():
    ref = np.array([np.nan, np.inf, -np.inf, 1.0])
    assert gate.allclose("t", ref.copy(), ref, "float16").passed
    for bad in ([0.0, np.inf, -np.inf, 1.0], [np.nan, -np.inf, -np.inf, 1.0], [np.nan, np.inf, -np.inf, np.nan]):
        assert gate.allclose("t", np.array(bad), ref, "float16").failing == 1


# --------------------------------------------------------------------------- #
# growth of a reduction's error with its length
# --------------------------------------------------------------------------- #
def _series(name, law, lengths=(256, 1024, 4096, 16384), seeds=3, bias=0.0, N=512):
    s = growth.Series(name)
    rng = np.random.default_rng(7)
    for T in lengths:
        for seed in range(seeds):
            gold = rng.standard_normal(N)
            err = law(T) * rng.standard_normal(N) + bias * law(T)
            s.add(T, seed, gold + err, gold)
    return s


def test_growth_laws_are_classified():
    sq = _series("sqrt", lambda T: 1e-8 * np.sqrt(T))
    lin = _series("linear", lambda T: 1e-10 * T)
    assert sq.exponent() == pytest.approx(0.5, abs=0.05)
    assert lin.exponent() == pytest.approx(1.0, abs=0.05)
    assert growth.growth_class(sq.exponent()) == "sqrt(T)-like"
    assert growth.growth_class(lin.exponent()) == "T-like"


def test_judge_accepts_the_same_envelope_and_rejects_bias_and_faster_growth():
    ref = _series("reference", lambda T: 1e-8 * np.sqrt(T))
    same = _series("target", lambda T: 0.7e-8 * np.sqrt(T))
    assert growth.judge(same, ref).verdict == "PASS WITH LIMITATIONS"
    biased = _series("target", lambda T: 0.7e-8 * np.sqrt(T), bias=1.0)
    assert growth.judge(biased, ref).verdict == "FAIL"
    faster = _series("target", lambda T: 1e-10 * T)
    assert growth.judge(faster, ref).verdict == "FAIL"
    single = _series("target", lambda T: 1e-8, lengths=(1024,))
    assert growth.judge(single, ref).verdict == "INCONCLUSIVE"


def test_oracle_orders_behave_as_summation_theory_says():
    """The oracle's two fp32 dgamma orders over growing M: the left-to-right sum
    has zero-mean rounding whose relative error grows like sqrt(M); the
    pairwise tree's barely grows."""
    seq, pw = growth.Series("sequential"), growth.Series("pairwise")
    for T in (256, 1024, 4096):
        for seed in range(2):
            x, g, dy = inputs.make_inputs(T, 128, "float32", seed=seed)
            _, gold = orc.bwd_golden(dy, x, g, "float32", want_dx=False)
            _, ref = orc.bwd_reference(dy, x, g, "float32", want_dx=False)
            seq.add(T, seed, ref, gold)
            pw.add(T, seed, orc.dgamma_pairwise_reference(dy, x, g, "float32"), gold)
    assert 0.3 < seq.exponent() < 0.7
    assert pw.exponent() < 0.25
    assert growth.judge(pw, seq).verdict == "PASS WITH LIMITATIONS"
