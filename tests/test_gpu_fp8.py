"""GPU parity of the 8-bit (E4M3) KV path against the CPU oracle.

K and V (cache and the step's own rows) are E4M3 codes read as code *
k_scale / code * v_scale; q and the output are bf16.  Outputs must match the
oracle within the bf16 tolerance 2e-2 (every output on small cases, a seeded
sample at full size); the fused step must append the accepted rows' codes bit
for bit.  Source: the speculative-sampling paper, end of section "Modified
rejection sampling" (the method composes with quantization); shapes as in the
BASS and EMS-SD abstracts.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import DeviceStep, compare_sampling, host_bits

pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module")
def api():
    import speculative_decoding_verify_09_gb300 as pkg
    pkg.build()
    return pkg.load()


def e4m3_inputs(name, with_logits=False, **kw):
    kw.setdefault("kv_dtype", "e4m3")
    inp = W.make_inputs(W.workload(name, **kw), with_logits=with_logits)
    assert inp["k_cache"].dtype == np.uint8
    return inp


def run_attn(api, inp):
    d = DeviceStep({k: v for k, v in inp.items()
                    if k not in ("target_logits", "draft_logits", "draft_tokens")}, api)
    api.spec_verify_attn(d.attn, d.ws)
    torch.cuda.synchronize()
    return d


def oracle_all(inp):
    return oracle.verify_attention(inp["q"], inp["k_new"], inp["v_new"], inp["k_cache"],
                                   inp["v_cache"], inp["cu_q"], inp["kv_start"], inp["kv_len"],
                                   inp["num_kv_heads"], k_scale=inp["k_scale"],
                                   v_scale=inp["v_scale"])


def full_check(api, inp):
    d = run_attn(api, inp)
    got = d.out.float().cpu().numpy()
    assert np.all(np.isfinite(got)), "unwritten or non-finite outputs"
    err = float(np.max(np.abs(got - oracle_all(inp))))
    assert err < TOL, err
    assert d.status_bits() == 0
    return d


@pytest.mark.parametrize("Hq,Hkv,K_hi", [
    (4, 4, 5),      # MHA, up to 6 rows (one 8-row group)
    (8, 4, 7),      # GQA g = 2, up to 16 packed rows
    (4, 4, 15),     # MHA, 16 block rows
])
def test_e4m3_small_all_outputs(api, Hq, Hkv, K_hi):
    full_check(api, e4m3_inputs("bass_b8", B=5, Hq=Hq, Hkv=Hkv, L_lo=0, L_hi=700, K_lo=0,
                                K_hi=K_hi, gen_seed=70 + K_hi))


def test_e4m3_q_range(api):
    """q is rounded to f16 for the tensor cores: inside the f16 range (here
    |q| up to ~6e4) the outputs match the oracle; one element beyond it makes
    only its own (row, head) output non-finite, as the header states."""
    inp = e4m3_inputs("bass_b8", B=3, Hq=4, Hkv=4, L_lo=10, L_hi=300, K_lo=1, K_hi=4,
                      gen_seed=83)
    q = W.bf16_bits_to_f32(inp["q"])
    q *= np.float32(6e4 / np.max(np.abs(q)))
    inp["q"] = W.f32_to_bf16_bits(q)
    inp.update(k_scale=6.25e-6, v_scale=0.0625)   # scores and outputs stay O(1)
    full_check(api, inp)
    r, h = 2, 1
    q2 = q.copy()
    q2[r, h, 7] = 7.0e4                        # beyond the f16 range
    inp["q"] = W.f32_to_bf16_bits(q2)
    d = run_attn(api, inp)
    got = d.out.float().cpu().numpy()
    ref = oracle_all(inp)
    bad = ~np.isfinite(got)
    assert bad[r, h].all()
    bad[r, h] = False
    assert not bad.any()
    mask = np.ones(got.shape[:2], dtype=bool)
    mask[r, h] = False
    assert float(np.max(np.abs(got[mask] - ref[mask]))) < TOL


def test_e4m3_scales_enter_as_defined(api):
    """k_scale scales the scores and v_scale the output: other scales on the
    same codes still match the oracle's definition."""
    inp = e4m3_inputs("bass_b8", B=3, Hq=4, Hkv=4, L_lo=10, L_hi=300, K_lo=1, K_hi=4,
                      gen_seed=81)
    inp.update(k_scale=0.03125, v_scale=0.5)
    full_check(api, inp)


def test_e4m3_one_long_sequence_many_pieces(api):
    full_check(api, e4m3_inputs("bass_b8", B=1, Hq=2, Hkv=1, L_lo=40000, L_hi=40000, K_lo=5,
                                K_hi=5, gen_seed=83))


def test_e4m3_full_size_sampled(api):
    inp = e4m3_inputs("bass_b8")
    d = run_attn(api, inp)
    got = d.out.float().cpu().numpy()
    assert np.all(np.isfinite(got))
    rng = np.random.default_rng(1)
    cu = inp["cu_q"]
    worst = 0.0
    for _ in range(96):
        i = int(rng.integers(0, inp["B"]))
        j = int(rng.integers(0, cu[i + 1] - cu[i]))
        h = int(rng.integers(0, inp["num_q_heads"]))
        ref = oracle.attention_row(i, h, j, inp["q"], inp["k_new"], inp["v_new"], inp["k_cache"],
                                   inp["v_cache"], cu, inp["kv_start"], inp["kv_len"],
                                   inp["num_kv_heads"], k_scale=inp["k_scale"],
                                   v_scale=inp["v_scale"])
        worst = max(worst, float(np.max(np.abs(got[cu[i] + j, h] - ref))))
    assert worst < TOL, worst
    assert d.status_bits() == 0


def test_e4m3_deterministic(api):
    inp = e4m3_inputs("bass_b8", B=6, L_lo=300, L_hi=3000, gen_seed=85)
    a = run_attn(api, inp).out.view(torch.int16).cpu()
    b = run_attn(api, inp).out.view(torch.int16).cpu()
    assert torch.equal(a, b)


def test_e4m3_fused_step(api):
    """Fused step over an E4M3 cache: decisions as the oracle's, accepted rows'
    codes appended bit for bit, attention within tolerance."""
    inp = e4m3_inputs("bass_b8", with_logits=True, B=6, Hq=8, Hkv=8, V=3000, L_lo=40,
                      L_hi=600, gen_seed=87)
    d = DeviceStep(inp, api)
    api.spec_verify_step(d.attn, d.sample, d.kv_cap, d.new_kv_len, d.ws)
    torch.cuda.synchronize()
    ref_s = oracle.reject_sample(inp["target_logits"], inp["draft_logits"], inp["draft_tokens"],
                                 inp["cu_q"], inp["kv_len"], inp["temperature"], inp["top_p"],
                                 inp["seed"], inp["seq_ids"])
    na = d.num_accepted.cpu().numpy()
    compare_sampling(ref_s, na, d.out_tokens.cpu().numpy(), inp["cu_q"])
    k2, v2, nl, st = oracle.kv_append(inp["k_cache"], inp["v_cache"], inp["k_new"], inp["v_new"],
                                      inp["cu_q"], inp["kv_start"], inp["kv_len"], inp["kv_cap"],
                                      na)
    assert np.array_equal(d.new_kv_len.cpu().numpy(), nl)
    assert np.array_equal(host_bits(d.k_cache), k2) and np.array_equal(host_bits(d.v_cache), v2)
    err = float(np.max(np.abs(d.out.float().cpu().numpy() - oracle_all(inp))))
    assert err < TOL, err
    assert d.status_bits() == (ref_s["status"] | st)


def test_e4m3_append_alone(api):
    inp = e4m3_inputs("bass_b8", with_logits=False, B=5, Hq=4, Hkv=4, L_lo=5, L_hi=80,
                      gen_seed=89)
    d = DeviceStep(inp, api)
    na = torch.tensor([0, 3, -1, 4, 1], dtype=torch.int32, device="cuda")
    na = torch.minimum(na, torch.from_numpy(np.diff(inp["cu_q"]) - 1).cuda())
    api.kv_append_ragged(d.cu_q, d.k_new, d.v_new, d.k_cache, d.v_cache, d.kv_start, d.kv_len,
                         d.kv_cap, na, d.new_kv_len, max_q_rows=d.max_q_rows,
                         dev_status=d.status)
    torch.cuda.synchronize()
    k2, v2, nl, _ = oracle.kv_append(inp["k_cache"], inp["v_cache"], inp["k_new"], inp["v_new"],
                                     inp["cu_q"], inp["kv_start"], inp["kv_len"], inp["kv_cap"],
                                     na.cpu().numpy())
    assert np.array_equal(d.new_kv_len.cpu().numpy(), nl)
    assert np.array_equal(host_bits(d.k_cache), k2) and np.array_equal(host_bits(d.v_cache), v2)


def test_e4m3_draft_positions(api):
    """Three draft positions (single-row attention, append of the row, draft
    draw) over an E4M3 cache against the oracle's draft_step with the scales."""
    from speculative_decoding_verify_09_gb300.buffers import DraftBuffers
    w = W.workload("bass_b8", B=6, L_lo=100, L_hi=900, kv_dtype="e4m3", gen_seed=91)
    base, steps = W.make_draft_inputs(w, positions=3)
    assert all(st["k_new"].dtype == np.uint8 for st in steps)
    d = DraftBuffers(base, api, positions=3, steps=steps)
    inp = dict(base)
    for t, st in enumerate(steps):
        inp.update(st)
        d.run()
        torch.cuda.synchronize()
        ref = oracle.draft_step(inp)
        err = float(np.max(np.abs(d.out[t].float().cpu().numpy() - ref["out"])))
        assert err < TOL, err
        got = d.tokens[t].cpu().numpy()
        for i in range(w.B):
            if not ref["tie"][i]:
                assert int(got[i]) == int(ref["tokens"][i])
        assert np.array_equal(host_bits(d.k_cache), ref["k_cache"])
        assert list(d.kv_len.cpu().numpy()) == list(ref["new_kv_len"])
        inp.update(k_cache=ref["k_cache"], v_cache=ref["v_cache"], kv_len=ref["new_kv_len"])
