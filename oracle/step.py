"""The fused verify step: attention, rejection sampling, ragged append.

TEST INFRASTRUCTURE ONLY: part of the CPU oracle.  Only tests, the smoke check
and the bench's CPU-baseline leg may import it.

Composition of the three parts, as one speculative-sampling loop iteration of
"Accelerating Large Language Model Decoding with Speculative Sampling"
(sections "Conditional scoring" and "Modified rejection sampling") over a
padding-free batch ("EMS-SD" and "BASS" abstracts).  The attention output and
the sampling decisions do not depend on each other inside one step (the logits
are inputs); the append depends on the decisions only.
"""
from .attention import verify_attention
from .sampling import reject_sample
from .append import kv_append


def verify_step(inp, attention=True):
    """Run the whole step on an input dict (see workloads.make_inputs).

    Returns a dict with out (float64 [R, Hq, D] or None), num_accepted,
    out_tokens, new_kv_len, k_cache, v_cache, status, seq_status and the
    near-tie audit of oracle.sampling.reject_sample.
    """
    prefix = None
    if inp.get("group") is not None:
        prefix = (inp["group"], inp["prefix_start"], inp["prefix_len"])
    out = None
    if attention:
        out = verify_attention(inp["q"], inp["k_new"], inp["v_new"], inp["k_cache"],
                               inp["v_cache"], inp["cu_q"], inp["kv_start"],
                               inp["kv_len"], inp["num_kv_heads"], inp.get("scale"),
                               prefix, inp.get("k_scale", 1.0), inp.get("v_scale", 1.0))
    s = reject_sample(inp["target_logits"], inp["draft_logits"], inp["draft_tokens"],
                      inp["cu_q"], inp["kv_len"], inp["temperature"], inp["top_p"],
                      inp["seed"], inp.get("seq_ids"), inp.get("top_k", 0),
                      inp.get("temperatures"), inp.get("top_ps"), inp.get("top_ks"))
    kc, vc, new_len, st = kv_append(inp["k_cache"], inp["v_cache"], inp["k_new"],
                                    inp["v_new"], inp["cu_q"], inp["kv_start"],
                                    inp["kv_len"], inp["kv_cap"], s["num_accepted"])
    return dict(out=out, num_accepted=s["num_accepted"], out_tokens=s["out_tokens"],
                new_kv_len=new_len, k_cache=kc, v_cache=vc, status=s["status"] | st,
                seq_status=s["seq_status"], tie_row=s["tie_row"],
                tie_kind=s["tie_kind"], tie_alts=s["tie_alts"],
                tie_count=s["tie_count"], tie_clauses=s["tie_clauses"],
                tie_positions=s["tie_positions"])
