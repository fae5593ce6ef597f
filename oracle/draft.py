"""The draft side of one speculative-sampling loop, in float64.

TEST INFRASTRUCTURE ONLY: part of the CPU oracle.  Only tests, the smoke check
and the bench's CPU-baseline leg may import it.

Source: "Accelerating Large Language Model Decoding with Speculative Sampling"
(Chen et al.; SpS): the algorithm it states for speculative sampling has the
draft model propose K tokens one after another, each drawn from the draft
distribution p(. | context and the drafts so far), before the target scores
them; section "Modified rejection sampling", "compatibility with standard
sampling methods": temperature / top-k / nucleus change the probabilities
before the scheme, so a draft is drawn from the same processed row p_hat that
the accept rule later uses (Theorem 1 needs x~ ~ p_hat).  One draft position is
one decode step of the draft model over a padding-free batch ("EMS-SD" and
"BASS" abstracts): attention with a single query row per sequence over its
cache plus that row, append of the row, then the draw.

Readings (pages silent):
  * position: at a draft step the sequence's cache holds L rows and the step's
    own row sits at index L; the drawn token sits at index L + 1, the same index
    the verify step's row for that draft decides;
  * uniform: word 1 (the sampling word) of Philox4x32-10 at counter
    (L + 1, seq_id, stream 1), the stream the verify step never uses, so the
    draft token is independent of the verify step's accept and resample
    uniforms at the same index; the draw itself is the verify step's bonus draw
    (inverse CDF in index order, first x whose cumulative weight exceeds u * Z)
    on the processed draft row;
  * parameters and failures as in the verify step's sampling: invalid
    per-sequence parameters give NONFINITE | BAD_PARAM, a row with NaN or +inf or
    only -inf gives NONFINITE; a failed sequence gets token -1.
"""
import numpy as np

from .philox import verify_uniforms, STREAM_DRAFT
from .sampling import (process_row, sample_index, params_ok, to_f64, _cdf_margin,
                       DEV_NONFINITE, DEV_BAD_PARAM, TIE_EPS, NUCLEUS_TIE_EPS)
from .attention import verify_attention
from .append import kv_append


def draft_sample(draft_logits, kv_len, temperature, top_p, seed, seq_ids=None, top_k=0,
                 temperatures=None, top_ps=None, top_ks=None):
    """One draft token per sequence from its processed draft row.

    draft_logits [B, V] (stored float32 or bf16 bits), kv_len [B] the cache
    lengths before this position's append.  Returns dict with tokens [B] int32
    (-1 for a failed sequence), seq_status [B], status, and the near-tie audit:
    tie [B] bool (u within TIE_EPS of an end of the chosen token's CDF
    interval, or a nucleus boundary mass within NUCLEUS_TIE_EPS of top_p) and
    tie_alts {i: tokens a tied draw may also yield} for every tied sequence:
    the weighted tokens whose normalized CDF interval lies within TIE_EPS of u,
    and for a nucleus tie also those of the draw under the neighbouring cut.
    """
    B = int(np.asarray(kv_len).shape[0])
    kv_len = np.asarray(kv_len, dtype=np.int64)
    if seq_ids is None:
        seq_ids = np.arange(B, dtype=np.int64)
    tokens = np.full(B, -1, dtype=np.int32)
    seq_status = np.zeros(B, dtype=np.uint32)
    tie = np.zeros(B, dtype=bool)
    tie_alts = {}
    for i in range(B):
        T_i = temperature if temperatures is None else temperatures[i]
        tp_i = top_p if top_ps is None else top_ps[i]
        tk_i = top_k if top_ks is None else top_ks[i]
        if not params_ok(T_i, tp_i, tk_i):
            seq_status[i] = DEV_NONFINITE | DEV_BAD_PARAM
            continue
        row = process_row(to_f64(draft_logits[i]), T_i, tp_i, tk_i)
        if not row.valid:
            seq_status[i] = DEV_NONFINITE
            continue
        _, u = verify_uniforms(seed, seq_ids[i], np.int64(kv_len[i] + 1), STREAM_DRAFT)
        x = sample_index(row.probs, float(u))
        tokens[i] = x
        m, _, nb = _cdf_margin(row.probs, x, float(u))
        if m < TIE_EPS or row.margin < NUCLEUS_TIE_EPS:
            tie[i] = True
            alts = set(nb)
            if row.margin < NUCLEUS_TIE_EPS:
                alt = process_row(to_f64(draft_logits[i]), T_i, tp_i, tk_i, alt=True)
                xa = sample_index(alt.probs, float(u))
                _, _, nba = _cdf_margin(alt.probs, xa, float(u))
                alts |= set(nba)
            tie_alts[i] = alts
    status = int(np.bitwise_or.reduce(seq_status)) if B else 0
    return dict(tokens=tokens, seq_status=seq_status, status=status, tie=tie,
                tie_alts=tie_alts)


def draft_step(inp, attention=True):
    """One draft position for every sequence: attention of the single query row
    over cache rows [0, L) and itself, append of that row (L -> L + 1, skipped
    with the CAPACITY bit past kv_cap), and the draft draw at index L + 1.
    The append copies the step's own row and does not depend on the draw.

    inp: an input dict whose block has one row per sequence (cu_q = 0..B) and
    whose draft_logits hold one row per sequence.  Returns dict with out,
    tokens, new_kv_len, k_cache, v_cache, status, seq_status, tie, tie_alts.
    """
    out = None
    if attention:
        out = verify_attention(inp["q"], inp["k_new"], inp["v_new"], inp["k_cache"],
                               inp["v_cache"], inp["cu_q"], inp["kv_start"],
                               inp["kv_len"], inp["num_kv_heads"], inp.get("scale"), None,
                               inp.get("k_scale", 1.0), inp.get("v_scale", 1.0))
    s = draft_sample(inp["draft_logits"], inp["kv_len"], inp["temperature"], inp["top_p"],
                     inp["seed"], inp.get("seq_ids"), inp.get("top_k", 0),
                     inp.get("temperatures"), inp.get("top_ps"), inp.get("top_ks"))
    B = inp["B"]
    kc, vc, new_len, st = kv_append(inp["k_cache"], inp["v_cache"], inp["k_new"],
                                    inp["v_new"], inp["cu_q"], inp["kv_start"],
                                    inp["kv_len"], inp["kv_cap"], np.zeros(B, dtype=np.int32))
    return dict(out=out, tokens=s["tokens"], new_kv_len=new_len, k_cache=kc, v_cache=vc,
                status=s["status"] | st, seq_status=s["seq_status"], tie=s["tie"],
                tie_alts=s["tie_alts"])
