"""Acceptance efficiency against K (speculative-sampling paper, section on the
trade-off between longer drafts and more frequent scoring, Figure 1 middle:
mean accepted tokens per loop divided by K + 1 falls as K grows).

With drafts drawn from p_hat, row j of a sequence keeps its draft with
probability beta_j = sum_x min(p_hat_j(x), q_hat_j(x)) (Theorem 1's
acceptance), independently of the earlier rows' uniforms, and the loop stops at
the first rejection.  So the number of emitted tokens 1 + N has the survival
function P(N >= j) = prod_{t<j} beta_t, mean sum_{j=0..K} prod_{t<j} beta_t and
an exact variance from the same products.  The oracle's batched verify must
reproduce that mean within its sampling error, for every K; the curve itself
(mean emitted / (K + 1)) must fall with K when the betas are below one.
"""
import numpy as np
import pytest
from scipy.special import softmax

import oracle


def emitted_moments(betas):
    """Mean and variance of 1 + N for one sequence with row acceptances betas."""
    K = len(betas)
    s = np.concatenate([[1.0], np.cumprod(betas)])        # s[j] = P(N >= j)
    mean = s.sum()
    # E[(1 + N)^2] = 1 + 2 E[N] + E[N^2];  E[N^2] = sum_{j,k >= 1} s[max(j, k)]
    en = s[1:].sum()
    en2 = sum(s[max(j, k)] for j in range(1, K + 1) for k in range(1, K + 1))
    return mean, 1 + 2 * en + en2 - mean ** 2


def beta_of(q_logits, p_logits, T, top_p):
    q = oracle.process_row(q_logits, T, top_p).probs
    p = oracle.process_row(p_logits, T, top_p).probs
    return float(np.minimum(p, q).sum())


def test_moments_closed_form_by_enumeration():
    betas = [0.7, 0.4, 0.9]
    probs = {}
    for n in range(4):                         # N = n: first n kept, then a rejection (or the end)
        pr = np.prod(betas[:n]) * ((1 - betas[n]) if n < 3 else 1.0)
        probs[n] = pr
    mean = sum((1 + n) * p for n, p in probs.items())
    var = sum((1 + n) ** 2 * p for n, p in probs.items()) - mean ** 2
    m2, v2 = emitted_moments(betas)
    assert abs(m2 - mean) < 1e-12 and abs(v2 - var) < 1e-12


@pytest.mark.parametrize("K", [1, 3, 6])
def test_oracle_mean_emitted_matches_closed_form(K):
    rng = np.random.default_rng(100 + K)
    V, B, T, top_p = 40, 600, 1.0, 1.0
    # one (q, p) row pair per draft position, shared by all sequences
    ql = rng.normal(0, 1.5, size=(K + 1, V)).astype(np.float32)
    pl = (ql + rng.normal(0, 1.0, size=(K + 1, V))).astype(np.float32)
    betas = [beta_of(ql[j], pl[j], T, top_p) for j in range(K)]
    cu = (np.arange(B + 1) * (K + 1)).astype(np.int32)
    tgt = np.tile(ql, (B, 1))
    drf = np.tile(pl[:K], (B, 1))
    # drafts drawn from p_hat row by row (inverse CDF with this test's own RNG)
    drafts = np.empty(B * K, dtype=np.int32)
    for j in range(K):
        pj = softmax(pl[j].astype(np.float64) / T)
        drafts[j::K] = rng.choice(V, size=B, p=pj)
    res = oracle.reject_sample(tgt, drf, drafts, cu, rng.integers(0, 5000, size=B), T, top_p,
                               7 + K, np.arange(B, dtype=np.int64) + 11)
    emitted = res["num_accepted"] + 1
    mean, var = emitted_moments(betas)
    z = (emitted.mean() - mean) / np.sqrt(var / B)
    assert abs(z) < 5, (emitted.mean(), mean, z)


def test_efficiency_falls_with_k():
    betas = np.full(8, 0.65)
    eff = [emitted_moments(betas[:K])[0] / (K + 1) for K in range(1, 9)]
    assert all(a > b for a, b in zip(eff, eff[1:]))
    # geometric case: mean = (1 - b^(K+1)) / (1 - b)
    for K in range(1, 9):
        assert abs(emitted_moments(betas[:K])[0] - (1 - 0.65 ** (K + 1)) / 0.35) < 1e-12
