"""Pins of the oracle's modified rejection sampler against what the method fixes.

Source: "Accelerating Large Language Model Decoding with Speculative
Sampling" -- section "Modified rejection sampling" (accept with probability
min(1, q/p), stop at the first rejection, resample from (q-p)_+, bonus token,
1..K+1 tokens per loop) and appendix "Proof", Theorem 1 (the output law is q;
P(accept, X=x) = min(p(x), q(x)); P(reject) = sum_x max(0, q(x)-p(x))).

The oracle's decisions are driven by 24-bit uniforms u = k * 2^-24.  The
implementation law is therefore computed exactly by counting grid points with
bisection on the oracle's own (monotone) decision functions, treated as black
boxes, and the whole-step composition is taken from `verify_sequence` itself.
"""
from fractions import Fraction
import itertools

import numpy as np
import pytest
from scipy import stats

from oracle import sampling as S
from oracle.philox import verify_uniforms

GRID = 1 << 24


def grid_u(k):
    return k * 2.0 ** -24


def count_accepting(p_d, q_d):
    """# of grid u the oracle's accept() takes (it is monotone: accepted for
    all u below a threshold)."""
    lo, hi = 0, GRID          # invariant: accept(lo-1) true or lo == 0; find first reject
    while lo < hi:
        mid = (lo + hi) // 2
        if S.accept(grid_u(mid), p_d, q_d):
            lo = mid + 1
        else:
            hi = mid
    return lo


def draw_counts(weights):
    """# of grid u that the oracle's sample_index maps to each index."""
    V = len(weights)
    first = []                # first grid k whose draw index is >= x
    for x in range(V + 1):
        lo, hi = 0, GRID
        while lo < hi:
            mid = (lo + hi) // 2
            if S.sample_index(weights, grid_u(mid)) >= x:
                hi = mid
            else:
                lo = mid + 1
        first.append(lo)
    return [first[x + 1] - first[x] for x in range(V)], first


def rand_dist(rng, V, peaky=1.0):
    w = rng.gamma(peaky, size=V)
    return w / w.sum()


# ---------------------------------------------------------------- primitives
def test_accept_count_matches_min_ratio():
    rng = np.random.default_rng(1)
    for _ in range(300):
        p, q = rng.uniform(1e-6, 1, size=2)
        c = count_accepting(p, q)
        assert abs(c - GRID * min(1.0, q / p)) <= 1.0
    assert count_accepting(0.3, 0.3) == GRID          # p == q: always accept
    assert count_accepting(0.0, 0.2) == GRID          # p == 0 < q: accept
    assert count_accepting(0.0, 0.0) == 0             # p == q == 0: reject
    assert count_accepting(0.5, 0.0) == 0


def test_draw_counts_match_normalized_weights():
    rng = np.random.default_rng(2)
    for V in (2, 5, 8, 13):
        w = rand_dist(rng, V) * rng.uniform(0.1, 3)
        w[rng.integers(0, V)] = 0.0
        cnt, _ = draw_counts(w)
        ideal = GRID * w / w.sum()
        assert np.all(np.abs(np.array(cnt) - ideal) <= 1.0)
        assert all(c == 0 for c, wx in zip(cnt, w) if wx == 0)   # zero weight never drawn


def test_residual_is_positive_part():
    q = np.array([0.5, 0.1, 0.4, 0.0])
    p = np.array([0.2, 0.3, 0.4, 0.1])
    assert list(S.residual(q, p)) == [0.3, 0.0, 0.0, 0.0]
    # Theorem 1 identity: 1 - sum min(p, q) == sum max(0, q - p)
    rng = np.random.default_rng(3)
    for _ in range(50):
        p, q = rand_dist(rng, 16), rand_dist(rng, 16)
        assert abs((1 - np.minimum(p, q).sum()) - S.residual(q, p).sum()) < 1e-12


def test_sample_index_fraction_and_empty():
    w = np.array([Fraction(1, 3), Fraction(0), Fraction(2, 3)], dtype=object)
    assert S.sample_index(w, Fraction(1, 3)) == 2       # strict: C(0) = 1/3 not > 1/3
    assert S.sample_index(w, Fraction(1, 3) - Fraction(1, 10**9)) == 0
    assert S.sample_index(np.zeros(4), 0.5) is None


# ------------------------------------------------------- whole-step laws
def step_law(q_of, p_of, ctx, K, V, accept_w, draw_w):
    """Law of the tokens one step emits from context `ctx`, with the oracle's
    verify_sequence as the black box.  q_of(ctx) / p_of(ctx) give the
    processed rows; accept_w / draw_w turn primitive grid counts into weights.
    Returns {emitted tuple: weight}."""
    law = {}
    for drafts in itertools.product(range(V), repeat=K):
        pw = 1
        prefixes = [ctx + drafts[:j] for j in range(K + 1)]
        prows = [p_of(c) for c in prefixes[:K]]
        qrows = [q_of(c) for c in prefixes]
        for j in range(K):
            pw = pw * accept_w(prows[j][drafts[j]], 1)          # draft probability
        if pw == 0:
            continue
        qm = np.stack(qrows)
        pm = np.stack(prows) if K else np.zeros((0, V))
        for n in range(K + 1):
            # path: rows < n accept, row n rejects (or n == K: bonus)
            w_path = pw
            u_acc = np.zeros(K + 1)
            ok = True
            for j in range(n):
                c = count_accepting(prows[j][drafts[j]], qrows[j][drafts[j]])
                if c == 0:
                    ok = False
                    break
                w_path = w_path * accept_w(c, GRID)
                u_acc[j] = grid_u(0)
            if not ok:
                continue
            if n < K:
                c = count_accepting(prows[n][drafts[n]], qrows[n][drafts[n]])
                if c == GRID:
                    continue
                w_path = w_path * accept_w(GRID - c, GRID)
                u_acc[n] = grid_u(GRID - 1)
                weights = S.residual(qrows[n], prows[n])
            else:
                weights = qrows[K]
            cnt, first = draw_counts(weights)
            for x in range(V):
                if cnt[x] == 0:
                    continue
                u_smp = np.full(K + 1, grid_u(first[x]))
                n_out, tok, _ = S.verify_sequence(qm, pm, list(drafts), u_acc, u_smp)
                emitted = tuple(drafts[:n_out]) + (tok,)
                law[emitted] = law.get(emitted, 0) + w_path * draw_w(cnt[x], GRID)
    return law


def prefix_law(q_of, p_of, ctx, K, V, N, accept_w, draw_w, memo):
    """Law of the next N tokens from ctx, iterating steps."""
    key = (ctx, N)
    if key in memo:
        return memo[key]
    out = {}
    for e, w in step_law(q_of, p_of, ctx, K, V, accept_w, draw_w).items():
        if len(e) >= N:
            t = e[:N]
            out[t] = out.get(t, 0) + w
        else:
            for rest, w2 in prefix_law(q_of, p_of, ctx + e, K, V, N - len(e),
                                       accept_w, draw_w, memo).items():
                out[e + rest] = out.get(e + rest, 0) + w * w2
    memo[key] = out
    return out


def target_law(q_of, ctx, V, N):
    law = {}
    for toks in itertools.product(range(V), repeat=N):
        w = 1
        for k in range(N):
            w = w * q_of(ctx + toks[:k])[toks[k]]
        law[toks] = w
    return law


def _tables(seed, V, dyadic):
    rng = np.random.default_rng(seed)
    pool = []
    if dyadic:
        # p: powers of two summing to 1; q: multiples of 1/16 with the residual
        # mass a power of two / 16, so every accept threshold and every CDF
        # boundary sits exactly on the 2^-24 grid.
        while len(pool) < 12:
            parts = [1.0]
            while len(parts) < V and rng.random() < 0.8:
                k = int(rng.integers(0, len(parts)))
                h = parts.pop(k) / 2
                parts += [h, h]
            p = np.array(parts + [0.0] * (V - len(parts)))
            rng.shuffle(p)
            q = rng.multinomial(16, np.full(V, 1.0 / V)) / 16.0
            Z16 = S.residual(q, p).sum() * 16          # exact: dyadic values
            if Z16 in (1.0, 2.0, 4.0, 8.0) and p.sum() == 1.0:
                pool.append((p, q))
    else:
        for _ in range(12):
            pool.append((rand_dist(rng, V, 0.7), rand_dist(rng, V, 0.7)))

    def pick(ctx):
        return pool[hash((seed,) + tuple(ctx)) % len(pool)]
    return (lambda c: pick(c)[1]), (lambda c: pick(c)[0])


@pytest.mark.parametrize("V,K,N", [(4, 2, 3), (4, 3, 4), (8, 1, 2)])
def test_theorem1_exact_on_grid_aligned_tables(V, K, N):
    """Dyadic tables: the implemented law must equal prod q exactly."""
    q_of, p_of = _tables(100 + V * 10 + K, V, dyadic=True)
    fw = lambda a, b: Fraction(a) / b if b != 1 else Fraction(a)
    got = prefix_law(q_of, p_of, (), K, V, N, fw, fw, {})
    want = target_law(lambda c: [Fraction(x) for x in q_of(c)], (), V, N)
    want = {k: v for k, v in want.items() if v != 0}
    got = {k: v for k, v in got.items() if v != 0}
    assert got == want


@pytest.mark.slow
@pytest.mark.parametrize("V,K,N", [(8, 3, 1), (8, 2, 3), (4, 3, 4)])
def test_theorem1_general_tables_within_grid_bound(V, K, N):
    """Arbitrary tables: each decision's grid weight is within 2^-24 of its
    ideal probability, so each cell is within (decisions) * 2^-24."""
    q_of, p_of = _tables(7 + V + K, V, dyadic=False)
    fw = lambda a, b: a / b
    got = prefix_law(q_of, p_of, (), K, V, N, fw, fw, {})
    want = target_law(q_of, (), V, N)
    bound = 4 * (K + 2) * N * 2.0 ** -24
    for t, w in want.items():
        assert abs(got.get(t, 0.0) - w) <= bound + 1e-12, (t, got.get(t), w)


# ------------------------------------------------------------ special cases
def test_p_equals_q_accepts_everything_and_bonus_follows_q():
    rng = np.random.default_rng(4)
    V, K = 8, 4
    rows = np.stack([rand_dist(rng, V) for _ in range(K + 1)])
    drafts = [int(rng.integers(0, V)) for _ in range(K)]
    for k in (0, 12345, GRID - 1):
        n, tok, st = S.verify_sequence(rows, rows[:K], drafts, np.full(K + 1, grid_u(k)),
                                       np.full(K + 1, grid_u(k)))
        assert n == K and st == 0
        assert tok == S.sample_index(rows[K], grid_u(k))
    cnt, _ = draw_counts(rows[K])
    assert np.all(np.abs(np.array(cnt) - GRID * rows[K]) <= 1)


def test_one_hot_target_is_deterministic():
    V, K = 6, 3
    t = 4
    q = np.zeros(V)
    q[t] = 1.0
    p = np.full(V, 1.0 / V)
    for drafts in itertools.product(range(V), repeat=K):
        for k in (0, GRID // 3, GRID - 1):
            u = np.full(K + 1, grid_u(k))
            n, tok, _ = S.verify_sequence(np.stack([q] * (K + 1)), np.stack([p] * K),
                                          list(drafts), u, u)
            emitted = list(drafts[:n]) + [tok]
            assert all(e == t for e in emitted)


def test_one_hot_draft_accepts_with_prob_q_and_resamples_q_without_draft():
    rng = np.random.default_rng(6)
    V = 7
    q = rand_dist(rng, V)
    d = 2
    p = np.zeros(V)
    p[d] = 1.0
    assert abs(count_accepting(p[d], q[d]) - GRID * q[d]) <= 1
    cnt, _ = draw_counts(S.residual(q, p))
    want = q.copy()
    want[d] = 0
    want /= want.sum()
    assert np.all(np.abs(np.array(cnt) - GRID * want) <= 1)


def test_emitted_count_between_one_and_k_plus_one():
    rng = np.random.default_rng(7)
    V = 16
    for _ in range(300):
        K = int(rng.integers(0, 6))
        q = np.stack([rand_dist(rng, V, 0.5) for _ in range(K + 1)])
        p = np.stack([rand_dist(rng, V, 0.5) for _ in range(K)]) if K else np.zeros((0, V))
        drafts = [int(rng.integers(0, V)) for _ in range(K)]
        n, tok, _ = S.verify_sequence(q, p, drafts, rng.random(K + 1), rng.random(K + 1))
        assert 0 <= n <= K and 0 <= tok < V and q[n][tok] > 0


def test_bad_draft_token_is_a_rejection():
    V, K = 8, 2
    q = np.full((K + 1, V), 1.0 / V)
    n, tok, st = S.verify_sequence(q, q[:K], [3, 99], np.zeros(K + 1), np.full(K + 1, 0.5))
    assert n == 1 and st & S.DEV_BAD_TOKEN
    # q == p so the residual is empty: the draw falls back to q
    assert st & S.DEV_EMPTY_RESIDUAL and tok == 4


# ----------------------------------------------- closed form and chi-square
def test_acceptance_rate_matches_closed_form_with_philox():
    """P(accept) = sum_x min(p(x), q(x)) (Theorem 1), with the verify stream's
    uniforms and drafts drawn from p through the draft stream (1e6 draws)."""
    rng = np.random.default_rng(8)
    V = 32
    p, q = rand_dist(rng, V, 0.8), rand_dist(rng, V, 0.8)
    pos = np.arange(1, 1_000_001)
    u_acc, _ = verify_uniforms(42, 3, pos)
    u_drf, _ = verify_uniforms(42, 3, pos, stream=1)
    d = S.sample_index(p, u_drf)
    rate = np.mean(S.accept(u_acc, p[d], q[d]))
    want = np.minimum(p, q).sum()
    sd = np.sqrt(want * (1 - want) / pos.size)
    assert abs(rate - want) < 5 * sd


def _batch_logits(rng, V, B, K):
    # The same q/p rows for every sequence; sequences differ only by seq_id.
    zq = rng.normal(0, 1.5, size=(K + 1, V)).astype(np.float32)
    zp = (zq[:K] + rng.normal(0, 1.0, size=(K, V))).astype(np.float32)
    tgt = np.tile(zq, (B, 1))
    drf = np.tile(zp, (B, 1))
    cu = np.arange(B + 1, dtype=np.int32) * (K + 1)
    return zq, zp, tgt, drf, cu


def test_first_token_law_chi_square_through_batch_path():
    """First emitted token ~ q_hat row 0 (Theorem 1), through reject_sample
    with Philox uniforms; drafts drawn from p_hat with the draft stream."""
    rng = np.random.default_rng(9)
    V, B, K = 8, 20000, 2
    T, top_p = 0.9, 0.93
    zq, zp, tgt, drf, cu = _batch_logits(rng, V, B, K)
    qhat = [S.process_row(zq[j].astype(np.float64), T, top_p).probs for j in range(K + 1)]
    phat = [S.process_row(zp[j].astype(np.float64), T, top_p).probs for j in range(K)]
    # drafts for sequence i drawn left to right from p_hat (stream 1)
    toks = np.zeros((B, K), dtype=np.int32)
    for j in range(K):
        u, _ = verify_uniforms(0, np.arange(B), 7 + j + 1, stream=1)
        toks[:, j] = S.sample_index(phat[j], u)
    kv = np.full(B, 7, dtype=np.int32)
    r = S.reject_sample(tgt, drf, toks.reshape(-1), cu, kv, T, top_p, 0)
    first = r["out_tokens"][cu[:-1]]
    h = np.bincount(first, minlength=V)
    keep = qhat[0] > 0
    assert np.all(h[~keep] == 0)
    assert stats.chisquare(h[keep], B * qhat[0][keep]).pvalue > 1e-3
    # acceptance of row 0 vs the closed form
    acc0 = np.mean(r["num_accepted"] >= 1)
    want = np.minimum(qhat[0], phat[0]).sum()
    assert abs(acc0 - want) < 5 * np.sqrt(want * (1 - want) / B)


def test_positions_and_words_used_by_each_row():
    """Row j of sequence i decides token index kv_len+j+1: the accept test uses
    word 0 and the draw word 1 of Philox(seed, seq_id, kv_len+j+1)."""
    V, K, B = 16, 3, 64
    # q/p = 1/2 on every draft (p = 2 q there): accept iff u_acc < 1/2
    zp = np.zeros((K, V), dtype=np.float32)
    zp[:, 0] = np.log(2.0)
    zq = np.zeros((K + 1, V), dtype=np.float32)
    tgt = np.tile(zq, (B, 1))
    drf = np.tile(zp, (B, 1))
    cu = np.arange(B + 1, dtype=np.int32) * (K + 1)
    toks = np.zeros(B * K, dtype=np.int32)
    kv = np.arange(B, dtype=np.int32) * 13 + 5
    sids = np.arange(B, dtype=np.int64) * 1000003 + (1 << 40)
    r = S.reject_sample(tgt, drf, toks, cu, kv, 1.0, 1.0, 77, seq_ids=sids)
    for i in range(B):
        pos = kv[i] + np.arange(K + 1) + 1
        ua, us = verify_uniforms(77, sids[i], pos)
        # p_hat(0) = 2/(V+1), q_hat(0) = 1/V: ratio = (V+1)/(2V)
        ratio = (V + 1) / (2 * V)
        n = next((j for j in range(K) if not ua[j] < ratio), K)
        assert r["num_accepted"][i] == n
        if n == K:          # bonus: uniform q over V -> floor(u * V)
            assert r["out_tokens"][cu[i] + n] == int(us[n] * V)


def test_batch_equals_independent_sequences_and_order_free():
    """Padding-free batch == each sequence alone (EMS-SD abstract), and the
    result of a sequence depends on its seq_id, not its batch slot."""
    rng = np.random.default_rng(10)
    V = 40
    Ks = [0, 3, 1, 5, 2]
    B = len(Ks)
    cu = np.concatenate([[0], np.cumsum(np.array(Ks) + 1)]).astype(np.int32)
    R = int(cu[-1])
    tgt = rng.normal(0, 2, size=(R, V)).astype(np.float32)
    drf = rng.normal(0, 2, size=(R - B, V)).astype(np.float32)
    toks = rng.integers(0, V, size=R - B).astype(np.int32)
    kv = rng.integers(0, 100, size=B).astype(np.int32)
    sids = np.array([5, 1, 9, 3, 7], dtype=np.int64)
    full = S.reject_sample(tgt, drf, toks, cu, kv, 0.8, 0.9, 3, seq_ids=sids)
    for i in range(B):
        r0, r1 = cu[i], cu[i + 1]
        p0 = r0 - i
        one = S.reject_sample(tgt[r0:r1], drf[p0:p0 + Ks[i]], toks[p0:p0 + Ks[i]],
                              np.array([0, r1 - r0], dtype=np.int32), kv[i:i + 1],
                              0.8, 0.9, 3, seq_ids=sids[i:i + 1])
        assert one["num_accepted"][0] == full["num_accepted"][i]
        assert list(one["out_tokens"]) == list(full["out_tokens"][r0:r1])
        assert 1 <= full["num_accepted"][i] + 1 <= Ks[i] + 1


def test_nonfinite_row_fails_only_its_sequence():
    V = 8
    cu = np.array([0, 2, 4], dtype=np.int32)
    tgt = np.zeros((4, V), dtype=np.float32)
    drf = np.zeros((2, V), dtype=np.float32)
    tgt[1, 3] = np.nan
    r = S.reject_sample(tgt, drf, np.array([1, 2], dtype=np.int32), cu,
                        np.array([0, 0], dtype=np.int32), 1.0, 1.0, 0)
    assert r["num_accepted"][0] == -1 and list(r["out_tokens"][:2]) == [-1, -1]
    assert r["seq_status"][0] == S.DEV_NONFINITE and r["seq_status"][1] == 0
    assert r["num_accepted"][1] == 1        # p == q: accepted


def test_rows_after_the_first_rejection_cannot_fail():
    """Draft 1 is certain to be rejected (p puts all mass on it, q none), so
    the loop stops at pair 0: a NaN in pair 1 or in the bonus row is never
    read and the sequence succeeds; the same NaN in pair 0 fails it."""
    V = 8
    cu = np.array([0, 3], dtype=np.int32)
    tgt = np.zeros((3, V), dtype=np.float32)
    drf = np.zeros((2, V), dtype=np.float32)
    tgt[0, 5] = -np.inf                     # q(5) = 0
    drf[0, :] = -np.inf
    drf[0, 5] = 0.0                         # p one-hot at 5
    drafts = np.array([5, 1], dtype=np.int32)
    for r_bad in ("t1", "d1", "t2"):
        t, d = tgt.copy(), drf.copy()
        if r_bad == "t1":
            t[1, 0] = np.nan
        elif r_bad == "d1":
            d[1, 0] = np.inf
        else:
            t[2, :] = -np.inf
        r = S.reject_sample(t, d, drafts, cu, np.array([4], dtype=np.int32), 1.0, 1.0, 9)
        assert r["num_accepted"][0] == 0 and r["seq_status"][0] == 0, r_bad
        assert r["out_tokens"][0] not in (-1, 5) and list(r["out_tokens"][1:]) == [-1, -1]
    t = tgt.copy()
    t[0, 2] = np.nan
    r = S.reject_sample(t, drf, drafts, cu, np.array([4], dtype=np.int32), 1.0, 1.0, 9)
    assert r["num_accepted"][0] == -1 and r["seq_status"][0] == S.DEV_NONFINITE


# ---------------------------------------------------------------- processing
def test_temperature_only_is_library_softmax():
    from scipy.special import softmax
    rng = np.random.default_rng(12)
    for T in (1.0, 0.7, 1.9):
        l = rng.normal(0, 4, size=300).astype(np.float32).astype(np.float64)
        got = S.process_row(l, T, 1.0).probs
        want = softmax(l / float(np.float32(T)))
        assert np.max(np.abs(got - want)) < 1e-15


def _nucleus_by_sorting(z, top_p):
    """Brute force: sort descending, cut at the first cumulative mass >= top_p,
    then widen the cut to the whole tie class of the last kept value."""
    P = np.exp(z - z.max())
    P /= P.sum()
    order = sorted(range(len(z)), key=lambda x: -z[x])
    c = 0.0
    for k, x in enumerate(order):
        c += P[x]
        if c >= top_p:
            break
    cut = z[order[k]]
    return {x for x in range(len(z)) if z[x] >= cut}


def test_nucleus_matches_sorting_with_ties():
    from scipy.special import softmax
    rng = np.random.default_rng(13)
    for trial in range(200):
        V = int(rng.integers(2, 60))
        z = rng.integers(-6, 6, size=V).astype(np.float64) * 0.5     # many ties
        top_p = float(np.float32(rng.uniform(0.05, 0.999)))
        row = S.process_row(z, 1.0, top_p)
        keep = set(np.flatnonzero(row.probs > 0).tolist())
        if row.margin < 1e-9:
            continue                       # mass exactly at top_p: rounding-defined
        assert keep == _nucleus_by_sorting(z, top_p)
        kk = sorted(keep)
        assert np.allclose(row.probs[kk], softmax(z[kk]), rtol=1e-13, atol=0)
        # invariants: kept mass >= top_p; dropping the lowest kept class < top_p
        P = softmax(z)
        assert P[kk].sum() >= top_p
        low = min(z[kk])
        assert P[[x for x in kk if z[x] > low]].sum() < top_p


def test_top_p_one_is_identity_and_minus_inf_is_masked():
    z = np.array([0.0, -np.inf, 1.0, -np.inf])
    r = S.process_row(z, 1.0, 1.0)
    assert r.valid and r.probs[1] == 0 and r.probs[3] == 0
    assert abs(r.probs.sum() - 1) < 1e-15
    assert not S.process_row(np.full(4, -np.inf), 1.0, 1.0).valid
    assert not S.process_row(np.array([0.0, np.inf]), 1.0, 0.9).valid


# --------------------------------------------------------------------------
# greedy, top-k and per-sequence parameters (SpS, "compatibility with
# standard sampling methods": the transforms apply before the scheme)
# --------------------------------------------------------------------------
def _topk_by_sorting(z, k):
    """Keep the k largest values, ties at the boundary kept, by full sort."""
    order = sorted(range(len(z)), key=lambda x: -z[x])
    thresh = z[order[k - 1]]
    return np.array([zz >= thresh for zz in z])


@pytest.mark.parametrize("k", [1, 2, 5, 17, 99, 100, 150])
def test_top_k_matches_sorting_with_ties(k):
    rng = np.random.default_rng(k)
    for T in (1.0, 0.7):
        l = rng.integers(-6, 6, size=100).astype(np.float64) * 0.5     # heavy ties
        l[rng.integers(0, 100, size=5)] = -np.inf
        r = S.process_row(l, T, 1.0, k)
        z = l / float(np.float32(T))
        if k < 100:
            keep = _topk_by_sorting(z, k)
        else:
            keep = np.ones(100, dtype=bool)
        w = np.where(keep, np.exp(z - z[np.isfinite(z)].max()), 0.0)
        assert np.allclose(r.probs, w / w.sum(), rtol=1e-12, atol=0)
        assert (r.probs > 0).sum() >= min(k, int(np.isfinite(l).sum()))


def test_top_k_then_top_p_is_nucleus_of_the_renormalized_top_k():
    rng = np.random.default_rng(5)
    for trial in range(20):
        l = rng.normal(0, 2, size=60)
        l[:10] = np.round(l[:10])                       # a few ties
        k, tp = int(rng.integers(1, 60)), float(np.float32(rng.uniform(0.1, 0.99)))
        r = S.process_row(l, 1.0, tp, k)
        keep = _topk_by_sorting(l, k)
        w = np.where(keep, np.exp(l - l.max()), 0.0)
        P = w / w.sum()
        nuc = _nucleus_by_sorting(np.where(keep, l, -np.inf), tp)
        want = np.where(np.isin(np.arange(len(l)), sorted(nuc)), P, 0.0)
        if r.margin > 1e-9:
            assert np.allclose(r.probs, want / want.sum(), rtol=1e-12, atol=0)


def test_greedy_row_is_one_hot_at_first_maximum():
    l = np.array([0.5, 3.0, -1.0, 3.0, 2.0, -np.inf])
    r = S.process_row(l, 0.0, 0.9, 3)
    assert r.valid and list(r.probs) == [0, 1, 0, 0, 0, 0]
    r = S.process_row(np.array([-np.inf, -np.inf]), 0.0, 1.0)
    assert not r.valid


def test_greedy_batch_keeps_drafts_equal_to_the_argmax_then_emits_it():
    """Closed form: with T = 0 a step keeps drafts while they equal the
    argmax of the target row, then emits the argmax of the first row that
    disagrees (or of the bonus row)."""
    rng = np.random.default_rng(8)
    B, V = 6, 40
    K = rng.integers(0, 5, size=B)
    cu = np.concatenate([[0], np.cumsum(K + 1)]).astype(np.int32)
    R = int(cu[-1])
    tgt = rng.integers(-5, 5, size=(R, V)).astype(np.float32)      # ties in the argmax
    src = np.concatenate([np.arange(cu[i], cu[i + 1] - 1) for i in range(B)])
    drf = tgt[src] + rng.integers(-1, 2, size=(R - B, V)).astype(np.float32)
    drafts = np.array([int(np.argmax(tgt[src[j]])) if rng.random() < 0.7 else
                       int(rng.integers(0, V)) for j in range(R - B)], dtype=np.int32)
    res = S.reject_sample(tgt, drf, drafts, cu, np.zeros(B, dtype=np.int32), 0.0, 1.0, 9)
    for i in range(B):
        r0, p0 = int(cu[i]), int(cu[i]) - i
        n = 0
        while n < K[i] and drafts[p0 + n] == int(np.argmax(tgt[r0 + n])):
            n += 1
        assert res["num_accepted"][i] == n
        assert list(res["out_tokens"][r0:r0 + n]) == list(drafts[p0:p0 + n])
        assert res["out_tokens"][r0 + n] == int(np.argmax(tgt[r0 + n]))


def test_per_sequence_parameters_equal_separate_batches():
    rng = np.random.default_rng(12)
    B, V = 5, 300
    _, _, tgt, drf, cu = _batch_logits(rng, V, B, 3)
    drafts = rng.integers(0, V, size=int(cu[-1]) - B).astype(np.int32)
    kv = rng.integers(0, 100, size=B).astype(np.int32)
    Ts = np.array([1.0, 0.0, 0.6, 1.3, 0.0], dtype=np.float32)
    tps = np.array([1.0, 0.9, 0.5, 0.95, 1.0], dtype=np.float32)
    tks = np.array([0, 0, 20, 5, 3], dtype=np.int32)
    seq_ids = np.arange(B, dtype=np.int64) + 40
    whole = S.reject_sample(tgt, drf, drafts, cu, kv, 1.0, 1.0, 77, seq_ids, 0, Ts, tps, tks)
    for i in range(B):
        r0, r1, p0 = int(cu[i]), int(cu[i + 1]), int(cu[i]) - i
        one = S.reject_sample(tgt[r0:r1], drf[p0:p0 + r1 - r0 - 1], drafts[p0:p0 + r1 - r0 - 1],
                              np.array([0, r1 - r0]), kv[i:i + 1], Ts[i], tps[i], 77,
                              seq_ids[i:i + 1], tks[i])
        assert whole["num_accepted"][i] == one["num_accepted"][0]
        assert list(whole["out_tokens"][r0:r1]) == list(one["out_tokens"])


def test_bad_per_sequence_parameters_fail_only_that_sequence():
    rng = np.random.default_rng(13)
    B, V = 4, 64
    _, _, tgt, drf, cu = _batch_logits(rng, V, B, 2)
    drafts = rng.integers(0, V, size=int(cu[-1]) - B).astype(np.int32)
    Ts = np.array([1.0, -1.0, np.nan, 1.0], dtype=np.float32)
    tps = np.array([1.0, 1.0, 1.0, 0.0], dtype=np.float32)
    res = S.reject_sample(tgt, drf, drafts, cu, np.zeros(B, dtype=np.int32), 1.0, 1.0, 1,
                          None, 0, Ts, tps, None)
    assert list(res["num_accepted"][1:]) == [-1, -1, -1] and res["num_accepted"][0] >= 0
    assert res["seq_status"][1] == S.DEV_NONFINITE | S.DEV_BAD_PARAM
    assert np.all(res["out_tokens"][cu[1]:] == -1)
