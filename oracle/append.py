"""Ragged KV append of the accepted rows only.

TEST INFRASTRUCTURE ONLY: part of the CPU oracle.  Only tests, the smoke check
and the bench's CPU-baseline leg may import it.

Source: "EMS-SD: Efficient Multi-sample Speculative Decoding" abstract: each
sample keeps its own number of accepted tokens with no padding tokens and no
extra memory.  Reading taken (bookkeeping the pages leave open): after n_i
acceptances, block rows 0..n_i of sequence i (the pending token and the n_i
accepted drafts) become committed, so n_i + 1 K/V rows are copied to cache rows
kv_start_i + L_i .. kv_start_i + L_i + n_i and the new length is L_i + n_i + 1.
The freshly sampled token is the next step's pending token.  If that would pass
the sequence's capacity kv_cap_i the append is skipped, the length stays L_i and
the CAPACITY status bit is set.  A sequence whose sampling failed (negative
num_accepted) is not appended.
"""
import numpy as np

from .sampling import DEV_CAPACITY


def kv_append(k_cache, v_cache, k_new, v_new, cu_q, kv_start, kv_len, kv_cap,
              num_accepted):
    """Returns (k_cache', v_cache', new_kv_len [B] int32, status bits)."""
    k_cache, v_cache = k_cache.copy(), v_cache.copy()
    B = len(cu_q) - 1
    new_len = np.asarray(kv_len, dtype=np.int32).copy()
    status = 0
    for i in range(B):
        n = int(num_accepted[i])
        if n < 0:
            continue
        L, cap, a, r0 = int(kv_len[i]), int(kv_cap[i]), int(kv_start[i]), int(cu_q[i])
        if L + n + 1 > cap:
            status |= DEV_CAPACITY
            continue
        k_cache[a + L:a + L + n + 1] = k_new[r0:r0 + n + 1]
        v_cache[a + L:a + L + n + 1] = v_new[r0:r0 + n + 1]
        new_len[i] = L + n + 1
    return k_cache, v_cache, new_len, status
