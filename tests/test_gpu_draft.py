"""GPU parity of the draft side against the CPU oracle (oracle/draft.py).

spec_draft_sample draws one token per sequence from the processed draft row
with Philox stream 1 at index kv_len + 1; tokens must match the oracle bit for
bit outside its near-tie windows (u within 1e-5 of an end of the chosen
token's CDF interval, nucleus boundary mass within 2e-6 of top_p), and inside
them be the oracle's token or one of its weighted neighbours.  A draft
position (single-row attention, append of the row, draw) is checked over
several consecutive positions: attention within 2e-2 (bf16) / 1e-4 (fp32),
caches, lengths and tokens exact.  Sources: "Accelerating Large Language Model
Decoding with Speculative Sampling", its speculative-sampling algorithm (draft
tokens drawn one at a time from p) and section "Modified rejection sampling"
(processing before the scheme); EMS-SD abstract (padding-free batches).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from speculative_decoding_verify_09_gb300.buffers import DraftBuffers, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    import speculative_decoding_verify_09_gb300 as pkg
    pkg.build()
    return pkg.load()


def compare_draft(ref, got):
    ties = 0
    for i, tok in enumerate(got):
        if ref["tie"][i]:
            ties += 1
            alts = ref["tie_alts"][i]
            assert int(tok) in alts, f"seq {i}: {tok} not in tie set {alts}"
            continue
        assert int(tok) == int(ref["tokens"][i]), f"seq {i}: {tok} != {ref['tokens'][i]}"
    return ties


def run_draw(api, base, seed=None):
    d = DraftBuffers(base, api, seed)
    api.spec_draft_sample(d.draft[0], d.ws_draft)
    torch.cuda.synchronize()
    return d, d.tokens[0].cpu().numpy()


def oracle_draw(base, seed=None):
    return oracle.draft_sample(base["draft_logits"], base["kv_len"], base["temperature"],
                               base["top_p"], base["seed"] if seed is None else seed,
                               base["seq_ids"], base.get("top_k", 0), base.get("temperatures"),
                               base.get("top_ps"), base.get("top_ks"))


def draft_inputs(name, **kw):
    base, _ = W.make_draft_inputs(W.workload(name, **kw))
    return base


@pytest.mark.parametrize("name,kw", [
    ("tiny_f32", {}),
    ("bass_b8", {}),
    ("bass_b8", dict(B=64, temperature=0.8, top_p=0.95)),
    ("bass_b8", dict(B=40, temperature=0.7, top_k=50)),
    ("bass_b8", dict(B=40, temperature=0.9, top_k=20, top_p=0.8)),
    ("bass_b8", dict(B=16, temperature=0.0)),
    ("ragged_gqa_b32", {}),
    ("vocab128k_b64", {}),
    ("vocab128k_b64", dict(temperature=1.0, top_p=1.0)),
])
def test_draft_sample_matches_oracle(api, name, kw):
    base = draft_inputs(name, **kw)
    ties = 0
    seeds = (0, 11, 2 ** 40 + 3)
    for seed in seeds:
        d, got = run_draw(api, base, seed)
        ref = oracle_draw(base, seed)
        ties += compare_draft(ref, got)
        assert d.status_bits() == ref["status"]
    # a draw is a tie with probability about sum_x min(p_hat(x), 2 * TIE_EPS)
    # (u within TIE_EPS of either end of the drawn token's interval): large
    # for long flat tails; the comparison must not be vacuous beyond that
    expect = len(seeds) * sum(
        np.minimum(oracle.process_row(oracle.to_f64(base["draft_logits"][i]),
                                      base["temperature"], base["top_p"],
                                      base.get("top_k", 0)).probs, 2 * oracle.TIE_EPS).sum()
        for i in range(base["B"]))
    assert ties <= 3 * expect + 3, (ties, expect)


def test_draft_sample_per_sequence_and_failures(api):
    base = draft_inputs("bass_b8", B=12)
    B = base["B"]
    lg = base["draft_logits"].copy()
    lg[3, 17] = 0x7FC0                                  # NaN (bf16 bits)
    lg[5, :] = 0xFF80                                   # all -inf
    base["draft_logits"] = lg
    base["temperatures"] = np.array([1.0, 0.0, 0.7, 1.0, 1.2, 1.0, -1.0, 0.5, 1.0, 0.9, 0.0, 1.0],
                                    dtype=np.float32)
    base["top_ps"] = np.array([1.0, 1.0, 0.9, 1.0, 0.5, 1.0, 1.0, 0.95, 0.0, 1.0, 0.3, 0.99],
                              dtype=np.float32)
    base["top_ks"] = np.array([0, 0, 0, 0, 10, 0, 0, 100, 0, 1, 5, 3], dtype=np.int32)
    d, got = run_draw(api, base)
    ref = oracle_draw(base)
    compare_draft(ref, got)
    assert list(got[[3, 5, 6, 8]]) == [-1, -1, -1, -1]
    assert d.status_bits() == ref["status"] == (oracle.DEV_NONFINITE | oracle.DEV_BAD_PARAM)
    assert all(got[i] >= 0 for i in range(B) if i not in (3, 5, 6, 8))


def test_draft_draws_use_their_own_stream(api):
    """Draft tokens for one batch equal the oracle's stream-1 draws and differ
    from what the verify stream's sampling word would pick on the same rows."""
    base = draft_inputs("bass_b8", B=64, V=64, temperature=1.0, logit_std=1.0)
    _, got = run_draw(api, base)
    ref = oracle_draw(base)
    compare_draft(ref, got)
    # the same rows drawn as bonus tokens of a K = 0 verify (stream 0)
    v = oracle.reject_sample(base["draft_logits"], base["draft_logits"][:0],
                             np.zeros(0, dtype=np.int32), base["cu_q"], base["kv_len"],
                             1.0, 1.0, base["seed"], base["seq_ids"])
    assert np.mean(v["out_tokens"] != got) > 0.5


@pytest.mark.parametrize("name,kw", [
    ("tiny_f32", {}),
    ("bass_b8", dict(B=6, L_lo=100, L_hi=900, temperature=0.8, top_p=0.9)),
    ("ragged_gqa_b32", dict(B=12, L_hi=3000)),
    ("bass_b8", {}),
])
@pytest.mark.parametrize("fused", [False, True])
def test_draft_positions_match_oracle(api, name, kw, fused):
    """Four consecutive draft positions through the C ABI (three calls per
    position, or the fused spec_draft_step) against the oracle's draft_step
    iterated: attention outputs, drawn tokens, appended rows and lengths after
    every position."""
    w = W.workload(name, **kw)
    base, steps = W.make_draft_inputs(w, positions=4)
    d = DraftBuffers(base, api, positions=4, steps=steps)
    inp = dict(base)
    tol = 1e-4 if w.dtype == "f32" else 2e-2
    for t, st in enumerate(steps):
        inp.update(st)
        d.run_fused() if fused else d.run()
        torch.cuda.synchronize()
        ref = oracle.draft_step(inp)
        err = float(np.max(np.abs(d.out[t].float().cpu().numpy() - ref["out"])))
        assert err <= tol, err
        compare_draft(ref, d.tokens[t].cpu().numpy())
        assert list(d.kv_len.cpu().numpy()) == list(ref["new_kv_len"])
        kc = host_bits(d.k_cache)
        vc = host_bits(d.v_cache)
        assert np.array_equal(kc, ref["k_cache"]) and np.array_equal(vc, ref["v_cache"])
        assert d.status_bits() == ref["status"]
        inp.update(k_cache=ref["k_cache"], v_cache=ref["v_cache"], kv_len=ref["new_kv_len"])


@pytest.mark.parametrize("fused", [False, True])
def test_draft_position_capacity_overflow(api, fused):
    base, _ = W.make_draft_inputs(W.workload("bass_b8", B=4, L_lo=64, L_hi=128))
    base = dict(base, kv_cap=base["kv_len"].copy())
    d = DraftBuffers(base, api)
    d.run_fused() if fused else d.run()
    torch.cuda.synchronize()
    assert list(d.kv_len.cpu().numpy()) == list(base["kv_len"])
    assert d.status_bits() & oracle.DEV_CAPACITY


@pytest.mark.parametrize("name,kw", [
    ("bass_b8", {}),
    ("ragged_gqa_b32", dict(B=16, L_hi=4000)),          # nucleus: the row-path sampler
])
def test_fused_draft_step_equals_three_calls(api, name, kw):
    """spec_draft_step gives the bits of the three separate calls (same
    kernels, same split of the attention, same Philox counters)."""
    base, steps = W.make_draft_inputs(W.workload(name, **kw), positions=3)
    a = DraftBuffers(base, api, positions=3, steps=steps)
    b = DraftBuffers(base, api, positions=3, steps=steps)
    a.run_all()
    b.run_all(fused=True)
    torch.cuda.synchronize()
    assert torch.equal(a.tokens, b.tokens)
    assert torch.equal(a.outputs["new_len"], b.outputs["new_len"])
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
    assert torch.equal(a.k_cache.view(torch.int16), b.k_cache.view(torch.int16))
    assert torch.equal(a.v_cache.view(torch.int16), b.v_cache.view(torch.int16))
    assert a.status_bits() == b.status_bits() == 0


def test_draft_step_rewinds_to_identical_results(api):
    """A whole draft-side step (every position from the starting lengths) run
    twice gives the same tokens, outputs and lengths: the starting lengths are
    never written and each position rewrites the same cache rows."""
    base, steps = W.make_draft_inputs(W.workload("bass_b8", B=8, L_hi=1000), positions=5)
    d = DraftBuffers(base, api, positions=5, steps=steps)
    d.run_all()
    torch.cuda.synchronize()
    first = (d.tokens.clone(), d.out.clone(), d.outputs["new_len"].clone())
    d.run_all()
    torch.cuda.synchronize()
    assert torch.equal(first[0], d.tokens) and torch.equal(first[2], d.outputs["new_len"])
    assert torch.equal(first[1].view(torch.int16), d.out.view(torch.int16))
    assert list(d.outputs["new_len"][-1].cpu().numpy()) == list(base["kv_len"] + 5)
