"""Pins of the oracle's draft side (oracle/draft.py) against what the pages and
the mathematics fix, independent of the oracle's own processing code:

* the law of the draft token is the processed draft distribution p_hat
  (softmax of logits / T, top-k, nucleus), computed here by sorting;
* SpS Theorem 1 end to end: drafts drawn by the draft sampler and verified by
  the verify sampler emit tokens with law q_hat even with a nucleus; drafts
  drawn from the unprocessed p break that law (the test has power);
* greedy drafting is the first argmax; a row with one finite entry draws it;
* failures stay with their sequence; one draft position appends exactly its
  row and later positions attend to it.
"""
import numpy as np
import pytest
from scipy import stats
from scipy.special import softmax

import oracle
import workloads as W


def _p_hat_by_sorting(l, T, top_p, top_k=0):
    """Processed distribution by full sort (ties at every cut kept)."""
    z = np.asarray(l, dtype=np.float64) / float(np.float32(T))
    order = np.argsort(-z, kind="stable")
    keep = np.ones(len(z), dtype=bool)
    if 0 < top_k < len(z):
        keep &= z >= z[order[top_k - 1]]
    P = np.where(keep, softmax(np.where(keep, z, -np.inf)), 0.0)
    tp = float(np.float32(top_p))
    if tp < 1.0:
        acc, cut = 0.0, None
        for x in order:
            if not keep[x]:
                continue
            acc += P[x]
            if acc >= tp:
                cut = z[x]
                break
        keep &= z >= cut
        P = np.where(keep, P, 0.0)
    return P / P.sum()


def _chi2_p(counts, probs):
    n = counts.sum()
    m = probs > 0
    assert counts[~m].sum() == 0, "a token outside the support was drawn"
    exp = probs[m] * n
    return stats.chisquare(counts[m], exp).pvalue


@pytest.mark.parametrize("T,top_p,top_k", [(1.0, 1.0, 0), (0.7, 0.8, 0), (1.3, 1.0, 4),
                                           (0.9, 0.9, 6)])
def test_draft_token_law_is_processed_p(T, top_p, top_k):
    rng = np.random.default_rng(int(T * 10) + top_k)
    V, N = 12, 12000
    l = rng.normal(0, 1.5, size=V)
    l[3] = l[7]                                       # a tie
    logits = np.tile(l.astype(np.float32), (N, 1))
    kv = rng.integers(0, 5000, size=N)
    res = oracle.draft_sample(logits, kv, T, top_p, 2024, np.arange(N) + 7, top_k)
    assert res["status"] == 0
    counts = np.bincount(res["tokens"], minlength=V)
    assert _chi2_p(counts, _p_hat_by_sorting(l.astype(np.float32), T, top_p, top_k)) > 1e-3


def _theorem1_run(draft_from_processed, top_p=0.6, T=1.0, N=10000):
    """First emitted token of N one-draft sequences sharing one (q, p) pair."""
    rng = np.random.default_rng(99)
    V = 8
    lq = rng.normal(0, 1.2, size=V).astype(np.float32)
    lp = (lq + rng.normal(0, 1.0, size=V)).astype(np.float32)
    kv = rng.integers(10, 4000, size=N)
    seq_ids = np.arange(N, dtype=np.int64) + 500
    if draft_from_processed:
        drafts = oracle.draft_sample(np.tile(lp, (N, 1)), kv, T, top_p, 77, seq_ids)["tokens"]
    else:                                   # control: ignores the nucleus
        pr = softmax(lp.astype(np.float64) / T)
        drafts = rng.choice(V, size=N, p=pr).astype(np.int32)
    cu = np.arange(0, 2 * N + 1, 2, dtype=np.int32)
    tgt = np.tile(lq, (2 * N, 1))
    res = oracle.reject_sample(tgt, np.tile(lp, (N, 1)), drafts, cu, kv, T, top_p, 77, seq_ids)
    first = res["out_tokens"][cu[:-1]]
    return np.bincount(first, minlength=V), _p_hat_by_sorting(lq, T, top_p)


def test_theorem1_through_draft_then_verify():
    counts, q_hat = _theorem1_run(True)
    assert _chi2_p(counts, q_hat) > 1e-3


def test_theorem1_control_unprocessed_drafts_break_the_law():
    counts, q_hat = _theorem1_run(False)
    m = q_hat > 0
    p = stats.chisquare(counts[m], q_hat[m] * counts[m].sum()).pvalue if counts[~m].sum() == 0 \
        else 0.0
    assert p < 1e-6


def test_greedy_draft_is_first_argmax_and_single_support_draws_it():
    l = np.array([[0.5, 3.0, -1.0, 3.0], [-np.inf, -np.inf, 2.0, -np.inf],
                  [1.0, 1.0, 1.0, 1.0]], dtype=np.float32)
    res = oracle.draft_sample(l, np.array([3, 9, 0]), 0.0, 1.0, 5)
    assert list(res["tokens"]) == [1, 2, 0]
    res = oracle.draft_sample(l[1:2], np.array([3]), 0.8, 0.5, 5)
    assert list(res["tokens"]) == [2]


def test_draft_failures_stay_with_their_sequence():
    rng = np.random.default_rng(4)
    l = rng.normal(size=(5, 30)).astype(np.float32)
    l[2, 4] = np.nan
    l[3, :] = -np.inf
    Ts = np.array([1.0, -0.5, 1.0, 1.0, 0.9], dtype=np.float32)
    res = oracle.draft_sample(l, np.zeros(5), 1.0, 1.0, 3, None, 0, Ts)
    assert list(res["tokens"][[1, 2, 3]]) == [-1, -1, -1]
    assert res["tokens"][0] >= 0 and res["tokens"][4] >= 0
    assert res["seq_status"][1] == oracle.DEV_NONFINITE | oracle.DEV_BAD_PARAM
    assert res["seq_status"][2] == oracle.DEV_NONFINITE == res["seq_status"][3]


def test_draft_positions_append_their_row_and_later_positions_see_it():
    """Three draft positions on the tiny workload: each appends its own K/V
    row at kv_start + L; the attention of position t equals the textbook
    softmax over the original cache rows, the rows appended before t and its
    own row (pure-Python scalar loops on fp64)."""
    w = W.workload("tiny_f32")
    base, steps = W.make_draft_inputs(w, positions=3)
    inp = dict(base)
    appended = []
    for t, st in enumerate(steps):
        inp.update(st)
        r = oracle.draft_step(inp)
        for i in range(inp["B"]):
            a, L = int(inp["kv_start"][i]), int(inp["kv_len"][i])
            assert r["new_kv_len"][i] == L + 1
            assert np.array_equal(r["k_cache"][a + L], st["k_new"][i])
            assert np.array_equal(r["v_cache"][a + L], st["v_new"][i])
            # textbook attention of sequence i, head 1, over every visible row
            L0 = int(base["kv_len"][i])
            keys = [base["k_cache"][a + x][1] for x in range(L0)] + \
                   [s["k_new"][i][1] for s in appended] + [st["k_new"][i][1]]
            vals = [base["v_cache"][a + x][1] for x in range(L0)] + \
                   [s["v_new"][i][1] for s in appended] + [st["v_new"][i][1]]
            qv = [float(x) for x in st["q"][i][1]]
            sc = [sum(qq * float(kk) for qq, kk in zip(qv, k)) / np.sqrt(w.D) for k in keys]
            m = max(sc)
            e = [np.exp(s - m) for s in sc]
            o = [sum(ee * float(v[d]) for ee, v in zip(e, vals)) / sum(e) for d in range(w.D)]
            assert np.allclose(r["out"][i][1], o, rtol=1e-12, atol=1e-12)
        appended.append(st)
        inp.update(k_cache=r["k_cache"], v_cache=r["v_cache"], kv_len=r["new_kv_len"])


def test_draft_capacity_overflow_keeps_length():
    base, _ = W.make_draft_inputs(W.workload("tiny_f32"))
    inp = dict(base, kv_cap=base["kv_len"].copy())
    r = oracle.draft_step(inp, attention=False)
    assert list(r["new_kv_len"]) == list(base["kv_len"])
    assert r["status"] & oracle.DEV_CAPACITY
