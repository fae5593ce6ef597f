"""The oracle against the hand-derived closed-form cases in tests/golden.

For each case the oracle's own decision functions are evaluated on the whole
24-bit uniform grid (by bisection, they are monotone): the keep probability of
a step, the normalized residual law and the law of the emitted token of a
one-draft step must equal the stored values exactly.  Source of the closed
forms: "Accelerating Large Language Model Decoding with Speculative Sampling",
section "Modified rejection sampling", appendix "Proof" (Theorem 1).
"""
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import sampling as S
from test_oracle_sampling import GRID, count_accepting, draw_counts, step_law

HERE = os.path.dirname(os.path.abspath(__file__))


def _cases():
    out = []
    for ln in open(os.path.join(HERE, "golden", "theorem1_cases.txt")):
        ln = ln.strip()
        if not ln or ln.startswith("#"):
            continue
        name, q, p, keep, res = [f.strip() for f in ln.split("|")]
        q = [Fraction(x) for x in q.split()]
        p = [Fraction(x) for x in p.split()]
        res = None if res == "-" else [Fraction(x) for x in res.split()]
        out.append((name, q, p, Fraction(keep), res))
    return out


CASES = _cases()


def test_fixture_is_well_formed():
    assert len(CASES) >= 7
    for name, q, p, keep, res in CASES:
        assert sum(q) == 1 and sum(p) == 1 and len(q) == len(p), name
        dyadic = lambda f: f.denominator & (f.denominator - 1) == 0
        assert all(dyadic(x) for x in q + p), name
        assert all(dyadic(qx / px) for qx, px in zip(q, p) if px > 0), name


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_keep_probability_and_residual(case):
    name, q, p, keep, res = case
    qf = np.array([float(x) for x in q])
    pf = np.array([float(x) for x in p])
    kept = sum(p[x] * Fraction(count_accepting(pf[x], qf[x]), GRID) for x in range(len(q)))
    assert kept == keep
    w = S.residual(qf, pf)
    if res is None:
        assert float(np.sum(w)) == 0.0
        return
    cnt, _ = draw_counts(w)
    assert [Fraction(c, GRID) for c in cnt] == res


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_emitted_token_law_is_q(case):
    """One-draft step through verify_sequence: the first emitted token has law q."""
    name, q, p, keep, res = case
    V = len(q)
    qf = np.array([float(x) for x in q])
    pf = np.array([float(x) for x in p])
    law = step_law(lambda c: qf, lambda c: pf, (), 1, V,
                   lambda a, b: Fraction(a) / Fraction(b) if b != 1 else Fraction(a),
                   lambda a, b: Fraction(a, b))
    first = [Fraction(0)] * V
    for toks, wgt in law.items():
        first[toks[0]] += wgt
    assert first == q
