"""Helpers for the GPU tests: compare the CUDA path with the oracle under
the near-tie rules.  Device buffers come from the package's StepBuffers."""
import numpy as np

from speculative_decoding_verify_09_gb300.buffers import StepBuffers as DeviceStep  # noqa: F401
from speculative_decoding_verify_09_gb300.buffers import dev, host_bits, to_f32  # noqa: F401


def compare_sampling(ref, num_accepted, out_tokens, cu_q):
    """Bit-exact comparison outside the oracle's near-tie windows.

    Returns (n_checked_sequences, n_tie_sequences).  Raises AssertionError with
    details on a mismatch."""
    B = len(cu_q) - 1
    ties = 0
    for i in range(B):
        r0, r1 = int(cu_q[i]), int(cu_q[i + 1])
        n_ref, n_gpu = int(ref["num_accepted"][i]), int(num_accepted[i])
        kind, row = int(ref["tie_kind"][i]), int(ref["tie_row"][i])
        if kind == 0:
            assert n_gpu == n_ref, f"seq {i}: num_accepted {n_gpu} != {n_ref}"
            assert list(out_tokens[r0:r1]) == list(ref["out_tokens"][r0:r1]), \
                f"seq {i}: tokens {list(out_tokens[r0:r1])} != {list(ref['out_tokens'][r0:r1])}"
            continue
        ties += 1
        if kind == 1:     # accept-level tie at `row`: rows before it still exact
            assert n_gpu >= row, f"seq {i}: gpu rejected at {n_gpu} before the tie row {row}"
            assert list(out_tokens[r0:r0 + row]) == list(ref["out_tokens"][r0:r0 + row])
        else:             # draw-level tie: n and accepted drafts exact, token a neighbour
            assert n_gpu == n_ref, f"seq {i}: num_accepted {n_gpu} != {n_ref} (draw tie)"
            assert list(out_tokens[r0:r0 + n_ref]) == list(ref["out_tokens"][r0:r0 + n_ref])
            alts = ref["tie_alts"].get(i)
            tok = int(out_tokens[r0 + n_ref])
            if alts is not None:
                assert tok in alts, f"seq {i}: drawn {tok} not in tie set {alts}"
            assert list(out_tokens[r0 + n_ref + 1:r1]) == [-1] * (r1 - r0 - n_ref - 1)
    return B, ties
