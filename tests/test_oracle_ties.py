"""Pins of the oracle's near-tie audit (what the GPU comparison may excuse).

The method ("Accelerating Large Language Model Decoding with Speculative
Sampling", section "Modified rejection sampling") fixes each decision exactly;
an fp32 path may differ only where a decision sits within the stated window of
its boundary: |u - min(1, q/p)| < 1e-5 at an accept test, or u within 1e-5 of
an end of the drawn token's normalized CDF interval.  These tests pin that the
audit flags exactly those decisions (brute force on small rows), that a draw
tie lists every token a 1e-5 CDF error can reach, that residuals of any mass
are audited the same way (no exemption for small residual mass), and the
neighbouring nucleus cut used for the nucleus clause.
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle.sampling import (TIE_EPS, NUCLEUS_TIE_EPS, TIE_ACCEPT, TIE_DRAW, _cdf_margin,
                             process_row, reject_sample, sample_index)


def _window_brute(weights, u):
    """Tokens with weight whose exact normalized CDF interval [lo, hi) meets
    [u - eps, u + eps], by a plain loop over Fractions."""
    w = [Fraction(float(x)) for x in weights]
    Z = sum(w)
    out, lo = set(), Fraction(0)
    U, E = Fraction(float(u)), Fraction(TIE_EPS)
    for i, x in enumerate(w):
        hi = lo + x / Z
        if x > 0 and hi > U - E and lo <= U + E:
            out.add(i)
        lo = hi
    return out


@pytest.mark.parametrize("seed", range(20))
def test_draw_window_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    V = int(rng.integers(2, 60))
    w = rng.exponential(size=V) * (rng.random(V) < 0.7)
    w[rng.integers(0, V)] += 1e-3
    # some tiny weights, narrower than the window
    w[rng.integers(0, V, size=3)] = 1e-9
    for u in list(rng.random(5)) + [0.0, 1.0 - 2 ** -24]:
        x = sample_index(w, u)
        m, Z, win = _cdf_margin(w, x, float(u))
        assert x in win
        assert win == _window_brute(w, u) | {x}
        c = np.cumsum(w) / Z
        lo = c[x - 1] if x else 0.0
        assert m == pytest.approx(min(u - lo, c[x] - u), abs=1e-15)


def test_small_residual_mass_is_audited_like_any_other():
    """A rejection whose residual sums to ~1e-6 is compared exactly unless its
    draw sits in the CDF window: no blanket exemption for small masses."""
    V = 64
    rng = np.random.default_rng(3)
    q_logits = rng.normal(0, 2, size=V)
    d = 5
    q_logits[d] = np.log(1e-6 / (np.exp(6.0) - 1.0)) + np.log(np.exp(q_logits).sum())
    p_logits = q_logits.copy()
    p_logits[d] += 6.0
    B = 40
    tgt = np.stack([q_logits, q_logits] * B).astype(np.float32)       # rows 0, 1 of each seq
    drf = np.stack([p_logits] * B).astype(np.float32)
    cu_q = np.arange(0, 2 * B + 1, 2, dtype=np.int32)
    drafts = np.full(B, d, dtype=np.int32)
    r = reject_sample(tgt, drf, drafts, cu_q, np.arange(B, dtype=np.int32) * 3, 1.0, 1.0, 0)
    rej = r["num_accepted"] == 0
    assert rej.sum() >= B // 2
    q = process_row(tgt[0].astype(np.float64), 1.0, 1.0).probs
    p = process_row(drf[0].astype(np.float64), 1.0, 1.0).probs
    Z = np.maximum(q - p, 0).sum()
    assert 3e-7 < Z < 3e-6
    for i in np.flatnonzero(rej):
        tok = int(r["out_tokens"][2 * i])
        assert tok != d                                 # outside the residual's support
        if r["tie_kind"][i] == 0:
            continue
        assert r["tie_kind"][i] == TIE_DRAW and tok in r["tie_alts"][i]
    assert r["tie_count"] < B // 4
    assert r["tie_clauses"]["cdf"] == r["tie_count"]


def test_accept_window_flags_only_close_decisions():
    """One draft, q/p = 1/2: u within 1e-5 of 1/2 is a tie, elsewhere not."""
    V = 4
    q = np.log(np.array([0.25, 0.25, 0.25, 0.25]))
    p = np.log(np.array([0.5, 0.5 / 3, 0.5 / 3, 0.5 / 3]))
    B = 3000
    tgt = np.stack([q, q] * B).astype(np.float64)
    drf = np.stack([p] * B).astype(np.float64)
    cu_q = np.arange(0, 2 * B + 1, 2, dtype=np.int32)
    from oracle.philox import verify_uniforms
    kv = np.arange(B, dtype=np.int32)
    r = reject_sample(tgt.astype(np.float32), drf.astype(np.float32),
                      np.zeros(B, dtype=np.int32), cu_q, kv, 1.0, 1.0, 11)
    ua, _ = verify_uniforms(11, np.arange(B), kv.astype(np.int64) + 1)
    q0 = process_row(tgt[0].astype(np.float32).astype(np.float64), 1.0, 1.0).probs[0]
    p0 = process_row(drf[0].astype(np.float32).astype(np.float64), 1.0, 1.0).probs[0]
    near = np.abs(ua - q0 / p0) < TIE_EPS
    got = (r["tie_kind"] == TIE_ACCEPT) & (r["tie_row"] == 0)
    assert np.array_equal(got, near)
    assert r["tie_clauses"]["accept"] == int(near.sum())


def test_nucleus_alternative_cut():
    """Five classes of masses 0.4, 0.3, 0.2, 0.06, 0.04 (one token each):
    top_p at the cumulative mass 0.9 of the first three +- a hair gives a
    boundary tie, and alt=True moves the cut by one class in the direction a
    rounding error could move it."""
    pr = np.array([0.4, 0.3, 0.2, 0.06, 0.04])
    l = np.log(pr)
    base = process_row(l, 1.0, 0.9 - 1e-7)       # reaches 0.9 with 3 classes
    assert base.margin < NUCLEUS_TIE_EPS
    assert np.count_nonzero(base.probs) == 3
    alt = process_row(l, 1.0, 0.9 - 1e-7, alt=True)
    assert np.count_nonzero(alt.probs) == 4      # "barely reaches": one class more
    base = process_row(l, 1.0, 0.7 + 1e-7)       # 0.7 barely missed by two classes
    assert np.count_nonzero(base.probs) == 3 and base.margin < NUCLEUS_TIE_EPS
    alt = process_row(l, 1.0, 0.7 + 1e-7, alt=True)
    assert np.count_nonzero(alt.probs) == 2
    far = process_row(l, 1.0, 0.8, alt=True)      # no tie: unchanged
    assert np.count_nonzero(far.probs) == 3 and far.margin > 1e-3
    assert np.allclose(alt.probs.sum(), 1.0)
