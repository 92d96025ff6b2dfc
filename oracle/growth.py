"""How the error of a column reduction grows with its length.

TEST INFRASTRUCTURE: see the package docstring. Pure numpy analysis of error
records; it computes no RMSNorm value itself.

Follows the page "torchtitan kernel numerics verification", section on the
analysis to run when the gate cannot be applied (the conditioning check's
alternative): repeat the reduction over several lengths T and several seeds;
an error that grows roughly like sqrt(T) is zero-mean rounding noise, one that
grows like T is a systematic bias; record the condition number at each T and
compare the distributions and the bias of the reference's and the target's
errors. Its verdict rules: both following the same conditioning-driven noise
envelope -> PASS WITH LIMITATIONS; a bias, abnormal scaling or semantic
mismatch of the target's own -> FAIL; evidence that cannot separate noise from
a bug -> INCONCLUSIVE.

Here it is a diagnostic for dgamma, the one reduction that runs over M rows
(up to 65,536 terms), where the gate itself is valid.

Readings of what the page leaves open (stated once, used throughout):
  * error at one (T, seed): the root mean square over the N columns of
    (result - golden), divided by the root mean square of golden, in fp64.
    Normwise relative, because an accumulation's rounding errors scale with
    its partial sums: a sum of T random-sign terms is ~sqrt(T) in size, so
    even a plain sequential sum's absolute error grows like T while its
    rounding stays zero-mean; relative to the result, that is sqrt(T), and a
    biased rounding (errors of one sign) grows like T. The growth exponent is
    the least-squares slope of log(error) against log(T) over every record;
  * "roughly sqrt(T)" vs "like T": an exponent below GROWTH_SPLIT (0.75, halfway)
    reads as sqrt(T)-like, at or above it as T-like;
  * the target follows the reference's envelope when its exponent is at most
    the reference's plus EXPONENT_SLACK and its error at every T is at most
    ENVELOPE_FACTOR times the reference's;
  * bias: the mean over columns of (result - golden) divided by its standard
    error (std / sqrt(N)); |z| > BIAS_Z at some T is a systematic bias when the
    reference shows none there.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

GROWTH_SPLIT = 0.75
EXPONENT_SLACK = 0.15
ENVELOPE_FACTOR = 2.0
BIAS_Z = 6.0


@dataclass
class Record:
    T: int
    seed: int
    rms_error: float
    bias_z: float


@dataclass
class Series:
    name: str
    records: list = field(default_factory=list)

    def add(self, T: int, seed: int, result, golden) -> Record:
        gold = np.asarray(golden, np.float64)
        d = np.asarray(result, np.float64) - gold
        scale = float(np.sqrt(np.mean(gold * gold)))
        rms = float(np.sqrt(np.mean(d * d))) / scale if scale > 0 else float("nan")
        sd = float(np.std(d))
        z = 0.0 if sd == 0.0 else float(np.mean(d) / (sd / np.sqrt(d.size)))
        rec = Record(int(T), int(seed), rms, z)
        self.records.append(rec)
        return rec

    def exponent(self) -> float:
        T = np.array([r.T for r in self.records], np.float64)
        e = np.array([r.rms_error for r in self.records], np.float64)
        keep = e > 0
        if keep.sum() < 2 or len(np.unique(T[keep])) < 2:
            return float("nan")
        return float(np.polyfit(np.log(T[keep]), np.log(e[keep]), 1)[0])

    def error_at(self, T: int) -> float:
        return float(np.median([r.rms_error for r in self.records if r.T == T]))

    def max_bias_z(self, T: int) -> float:
        return float(max(abs(r.bias_z) for r in self.records if r.T == T))


def growth_class(exponent: float) -> str:
    if not np.isfinite(exponent):
        return "undetermined"
    return "sqrt(T)-like" if exponent < GROWTH_SPLIT else "T-like"


@dataclass
class Verdict:
    verdict: str
    target_exponent: float
    reference_exponent: float
    notes: list


def judge(target: Series, reference: Series) -> Verdict:
    """The page's verdict for the target's growth against the reference's."""
    te, re_ = target.exponent(), reference.exponent()
    notes = [f"{target.name}: exponent {te:.2f} ({growth_class(te)}); "
             f"{reference.name}: exponent {re_:.2f} ({growth_class(re_)})"]
    if not (np.isfinite(te) and np.isfinite(re_)):
        return Verdict("INCONCLUSIVE", te, re_, notes + ["too few lengths or zero errors to fit"])
    lengths = sorted({r.T for r in target.records})
    failed = False
    for T in lengths:
        tb, rb = target.max_bias_z(T), reference.max_bias_z(T)
        if tb > BIAS_Z and rb <= BIAS_Z:
            failed = True
            notes.append(f"T={T}: target bias |z| = {tb:.1f} where the reference has {rb:.1f}")
        et, er = target.error_at(T), reference.error_at(T)
        if et > ENVELOPE_FACTOR * er:
            failed = True
            notes.append(f"T={T}: target error {et:.3e} above {ENVELOPE_FACTOR} x reference {er:.3e}")
    if te > re_ + EXPONENT_SLACK:
        failed = True
        notes.append(f"target grows faster than the reference ({te:.2f} > {re_:.2f} + {EXPONENT_SLACK})")
    if failed:
        return Verdict("FAIL", te, re_, notes)
    return Verdict("PASS WITH LIMITATIONS", te, re_, notes)


def report(title: str, series: list, conditions: dict, verdict: Verdict) -> str:
    """Markdown table: one row per length T (median over seeds)."""
    lengths = sorted({r.T for r in series[0].records})
    head = "| T | condition (median) | " + " | ".join(f"{s.name} rel rms err" for s in series) + \
           " | " + " | ".join(f"{s.name} max bias z" for s in series) + " |"
    sep = "|---" * (2 + 2 * len(series)) + "|"
    lines = [f"### {title}", head, sep]
    for T in lengths:
        lines.append(f"| {T} | {conditions.get(T, float('nan')):.3g} | "
                     + " | ".join(f"{s.error_at(T):.3e}" for s in series) + " | "
                     + " | ".join(f"{s.max_bias_z(T):.1f}" for s in series) + " |")
    for s in series:
        e = s.exponent()
        lines.append(f"- {s.name}: growth exponent {e:.2f} ({growth_class(e)})")
    lines += [f"- {n}" for n in verdict.notes]
    lines.append(f"Verdict: {verdict.verdict}")
    return "\n".join(lines)
