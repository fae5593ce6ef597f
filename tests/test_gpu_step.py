"""GPU parity of the fused spec_verify_step with the oracle's verify_step.

One call: verify attention, rejection sampling and the append of accepted
rows.  Tokens / accepted counts / appended rows / new lengths bit-exact
outside the near-tie windows; attention within 2e-2 (bf16) or 1e-4 (fp32);
pool rows the append must not touch stay identical.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import DeviceStep, compare_sampling, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    import speculative_decoding_verify_09_gb300 as pkg
    pkg.build()
    return pkg.load()


def run_step(api, inp):
    d = DeviceStep(inp, api)
    api.spec_verify_step(d.attn, d.sample, d.kv_cap, d.new_kv_len, d.ws)
    torch.cuda.synchronize()
    return d


def check_step(api, inp, attn_rows=None):
    d = run_step(api, inp)
    ref_s = oracle.reject_sample(inp["target_logits"], inp["draft_logits"], inp["draft_tokens"],
                                 inp["cu_q"], inp["kv_len"], inp["temperature"], inp["top_p"],
                                 inp["seed"], inp["seq_ids"], inp.get("top_k", 0),
                                 inp.get("temperatures"), inp.get("top_ps"), inp.get("top_ks"))
    na = d.num_accepted.cpu().numpy()
    _, ties = compare_sampling(ref_s, na, d.out_tokens.cpu().numpy(), inp["cu_q"])
    # append: checked against the oracle's append driven by the GPU's own
    # accepted counts (identical to the oracle's outside accept-level ties)
    exact = ref_s["tie_kind"] != oracle.TIE_ACCEPT
    assert np.array_equal(na[exact], ref_s["num_accepted"][exact])
    k2, v2, nl, st = oracle.kv_append(inp["k_cache"], inp["v_cache"], inp["k_new"], inp["v_new"],
                                      inp["cu_q"], inp["kv_start"], inp["kv_len"], inp["kv_cap"],
                                      na)
    assert np.array_equal(d.new_kv_len.cpu().numpy(), nl)
    assert np.array_equal(host_bits(d.k_cache), k2) and np.array_equal(host_bits(d.v_cache), v2)
    assert d.status_bits() == (ref_s["status"] | st)
    # attention
    got = d.out.float().cpu().numpy()
    assert np.all(np.isfinite(got))
    tol = 1e-4 if inp["dtype"] == "f32" else 2e-2
    cu = inp["cu_q"]
    rng = np.random.default_rng(0)
    prefix = None
    if inp.get("group") is not None:
        prefix = (inp["group"], inp["prefix_start"], inp["prefix_len"])
    if attn_rows is None:
        ref = oracle.verify_attention(inp["q"], inp["k_new"], inp["v_new"], inp["k_cache"],
                                      inp["v_cache"], cu, inp["kv_start"], inp["kv_len"],
                                      inp["num_kv_heads"], prefix=prefix)
        err = np.max(np.abs(got - ref))
    else:
        err = 0.0
        for _ in range(attn_rows):
            i = int(rng.integers(0, inp["B"]))
            j = int(rng.integers(0, cu[i + 1] - cu[i]))
            h = int(rng.integers(0, inp["num_q_heads"]))
            ref = oracle.attention_row(i, h, j, inp["q"], inp["k_new"], inp["v_new"],
                                       inp["k_cache"], inp["v_cache"], cu, inp["kv_start"],
                                       inp["kv_len"], inp["num_kv_heads"], prefix=prefix)
            err = max(err, float(np.max(np.abs(got[cu[i] + j, h] - ref))))
    assert err < tol, err
    return d, ties


def test_tiny_fp32_step(api):
    check_step(api, W.make_inputs(W.workload("tiny_f32")))


def test_small_bf16_step_all_outputs(api):
    check_step(api, W.make_inputs(W.workload("ragged_gqa_b32", B=6, V=3000, L_hi=900,
                                             gen_seed=31)))


@pytest.mark.parametrize("name", ["bass_b8", "ragged_gqa_b32", "vocab128k_b64",
                                  "shared_prefix_s32"])
def test_full_size_step(api, name):
    d, ties = check_step(api, W.make_inputs(W.workload(name)), attn_rows=64)
    print(name, "accepted", d.num_accepted.tolist()[:16], "tie sequences", ties)


def test_small_shared_prefix_step_all_outputs(api):
    check_step(api, W.make_inputs(W.workload("shared_prefix_s32", B=6, groups=2,
                                             prefix_lens=(200, 90), V=900, L_hi=100,
                                             gen_seed=33)))


def test_capacity_overflow_in_step(api):
    inp = W.make_inputs(W.workload("bass_b8", B=4, V=1000, L_hi=700, gen_seed=41))
    inp["kv_cap"] = inp["kv_len"] + 1          # room for the pending row only
    d, _ = check_step(api, inp)
    na = d.num_accepted.cpu().numpy()
    if np.any(na > 0):
        assert d.status_bits() & oracle.DEV_CAPACITY


def test_repeated_steps_are_identical(api):
    """Steps do not carry state: the workspace is left ready, lengths are
    separate outputs, so the same inputs give the same results."""
    inp = W.make_inputs(W.workload("ragged_gqa_b32", B=8, V=2000, L_hi=500, gen_seed=43))
    d = DeviceStep(inp, api)
    outs = []
    for _ in range(3):
        d.k_cache.copy_(torch.from_numpy(inp["k_cache"].view(np.int16)).cuda().view(torch.bfloat16))
        api.spec_verify_step(d.attn, d.sample, d.kv_cap, d.new_kv_len, d.ws)
        torch.cuda.synchronize()
        outs.append((d.out.clone(), d.out_tokens.clone(), d.new_kv_len.clone()))
    for o in outs[1:]:
        assert all(torch.equal(a, b) for a, b in zip(o, outs[0]))


def test_staged_step_one_copy_each_way(api):
    """Inputs in one pinned arena, one copy in, the fused call, one copy out:
    the host-side results equal the oracle's (same check as the plain path)."""
    from speculative_decoding_verify_09_gb300.buffers import StagedStep
    inp = W.make_inputs(W.workload("bass_b8", B=4, Hq=8, Hkv=8, V=2000, L_lo=50, L_hi=400,
                                   gen_seed=29))
    d = DeviceStep(inp, api)
    st = StagedStep(d)
    st.dev_in.zero_()                      # nothing left over from construction
    st.pack(inp)
    st.upload()
    api.spec_verify_step(st.attn, st.sample, d.kv_cap, d.new_kv_len, d.ws)
    st.download()
    torch.cuda.synchronize()
    ref = oracle.verify_step(inp)
    out = st.result("out").float().numpy()
    assert np.max(np.abs(out - ref["out"])) < 2e-2
    _, ties = compare_sampling(ref, st.result("num_accepted").numpy(),
                               st.result("out_tokens").numpy(), inp["cu_q"])
    if ties == 0:
        assert np.array_equal(st.result("new_kv_len").numpy(), ref["new_kv_len"])
    assert d.status_bits() == ref["status"]



def test_step_with_per_sequence_parameters(api):
    """Fused step on the row path (greedy / top-k / nucleus per sequence):
    decisions, appended rows and lengths as the oracle's."""
    inp = W.make_inputs(W.workload("bass_b8", B=6, Hq=8, Hkv=8, V=3000, L_lo=40, L_hi=300,
                                   gen_seed=51))
    inp["temperatures"] = np.array([0.0, 1.0, 0.7, 0.0, 1.2, 0.9], dtype=np.float32)
    inp["top_ps"] = np.array([1.0, 0.9, 1.0, 1.0, 0.6, 0.95], dtype=np.float32)
    inp["top_ks"] = np.array([0, 20, 5, 0, 0, 200], dtype=np.int32)
    check_step(api, inp)
