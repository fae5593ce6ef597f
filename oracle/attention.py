"""Verify attention over ragged KV caches, in float64.

TEST INFRASTRUCTURE ONLY: part of the CPU oracle.  Only tests, the smoke check
and the bench's CPU-baseline leg may import it.

Sources:
  * "Accelerating Large Language Model Decoding with Speculative Sampling",
    section "Conditional scoring" (条件评分): the target scores a K-token draft in
    one call; attention reads the KV cache of all earlier tokens, whose size
    does not change with K.
  * "BASS: Batched Attention-optimized Speculative Sampling" and "EMS-SD"
    abstracts: a batch of sequences with different lengths and different draft
    counts, handled without padding.
  * Bifurcated attention abstract (author page of Haifeng Qian): attention over
    a shared prefill KV plus a per-sample decode KV, split in two GEMMs, with a
    result that is precise, i.e. equal to attention over the concatenation.

8-bit KV (the speculative-sampling paper, end of section "Modified rejection
sampling": the method leaves the transformer body alone, so it combines with
memory-saving techniques such as quantization and multi-query attention): K/V
stored as E4M3 codes with per-tensor scales are read as code value times the
scale; the step's own block rows come in the same format as the cache (they
are written to it, then attended to).

Definition computed here (the plain one): for sequence i, query head h, block
row j, the keys/values are
    [shared prefix rows (bifurcated mode only)] ++ [cache rows kv_start_i ..
    kv_start_i + L_i - 1] ++ [draft-block rows 0..j]
with KV head h // (Hq / Hkv); out = softmax(scale * q . k) @ v, scale =
1/sqrt(D) unless given.  Readings: block row 0 is the pending token whose K/V
are not cached yet, rows 1..K_i are the drafts; causal inside the block.
"""
import numpy as np

from .sampling import to_f64


def _seq_keys(i, hk, k_cache, v_cache, kv_start, kv_len, prefix):
    ks, vs = [], []
    if prefix is not None:
        group, prefix_start, prefix_len = prefix
        g = int(group[i])
        a, n = int(prefix_start[g]), int(prefix_len[g])
        ks.append(k_cache[a:a + n, hk])
        vs.append(v_cache[a:a + n, hk])
    a, n = int(kv_start[i]), int(kv_len[i])
    ks.append(k_cache[a:a + n, hk])
    vs.append(v_cache[a:a + n, hk])
    return ks, vs


def attention_row(i, h, j, q, k_new, v_new, k_cache, v_cache, cu_q, kv_start,
                  kv_len, num_kv_heads, scale=None, prefix=None, k_scale=1.0, v_scale=1.0):
    """Output row (sequence i, head h, block row j) as a float64 [D] vector.

    K and V rows are the stored values times k_scale and v_scale (per-tensor
    dequantization scales of an 8-bit cache; 1 for bf16 / fp32 caches)."""
    Hq = q.shape[1]
    D = q.shape[2]
    hk = h // (Hq // num_kv_heads)
    if scale is None or scale == 0:
        scale = 1.0 / np.sqrt(D)
    r0 = int(cu_q[i])
    ks, vs = _seq_keys(i, hk, k_cache, v_cache, kv_start, kv_len, prefix)
    ks.append(k_new[r0:r0 + j + 1, hk])
    vs.append(v_new[r0:r0 + j + 1, hk])
    Kmat = to_f64(np.concatenate(ks, axis=0)) * float(np.float32(k_scale))
    Vmat = to_f64(np.concatenate(vs, axis=0)) * float(np.float32(v_scale))
    qv = to_f64(q[r0 + j, h])
    s = float(np.float32(scale)) * (Kmat @ qv)
    e = np.exp(s - s.max())
    return (e / e.sum()) @ Vmat


def verify_attention(q, k_new, v_new, k_cache, v_cache, cu_q, kv_start, kv_len,
                     num_kv_heads, scale=None, prefix=None, k_scale=1.0, v_scale=1.0):
    """All outputs, float64 [R, Hq, D].

    q [R, Hq, D]; k_new, v_new [R, Hkv, D]; k_cache, v_cache [P, Hkv, D] pools
    (token-major); cu_q [B+1]; kv_start [B]; kv_len [B]; prefix = (group [B],
    prefix_start [G], prefix_len [G]) or None.  Stored tensors are float32,
    bfloat16 bit patterns (uint16) or, for K and V, E4M3 codes (uint8) read as
    code value times k_scale / v_scale.
    """
    R, Hq, D = q.shape
    out = np.zeros((R, Hq, D))
    B = len(cu_q) - 1
    for i in range(B):
        for j in range(int(cu_q[i + 1]) - int(cu_q[i])):
            for h in range(Hq):
                out[int(cu_q[i]) + j, h] = attention_row(
                    i, h, j, q, k_new, v_new, k_cache, v_cache, cu_q, kv_start,
                    kv_len, num_kv_heads, scale, prefix, k_scale, v_scale)
    return out
