"""Helpers for the GPU tests: compare the CUDA path with the oracle under
the near-tie rules.  Device buffers come from the package's StepBuffers."""
import numpy as np

from speculative_decoding_verify_09_gb300.buffers import StepBuffers as DeviceStep  # noqa: F401
from speculative_decoding_verify_09_gb300.buffers import dev, host_bits, to_f32  # noqa: F401


def compare_sampling(ref, num_accepted, out_tokens, cu_q, drafts=None, V=None):
    """Bit-exact comparison outside the oracle's near-tie windows.

    Every sequence is checked: with no tie, n_i and all of its tokens exactly;
    with a tie at the final draw (TIE_DRAW), n_i and the accepted drafts
    exactly and the drawn token within the oracle's tie set (the weighted
    tokens whose normalized CDF interval lies within 1e-5 of u); with a tie at an accept decision or a
    nucleus cut (TIE_ACCEPT) at row r, the tokens before r exactly and the rest
    for validity (r <= n_i <= K_i, drafts kept in order when `drafts` is
    given, a drawn token in [0, V) when V is given, -1 after it).

    Returns (n_checked_sequences, n_tie_sequences).  Raises AssertionError with
    details on a mismatch."""
    B = len(cu_q) - 1
    ties = 0
    for i in range(B):
        r0, r1 = int(cu_q[i]), int(cu_q[i + 1])
        K = r1 - r0 - 1
        n_ref, n_gpu = int(ref["num_accepted"][i]), int(num_accepted[i])
        kind, row = int(ref["tie_kind"][i]), int(ref["tie_row"][i])
        got = [int(t) for t in out_tokens[r0:r1]]
        want = [int(t) for t in ref["out_tokens"][r0:r1]]
        if kind == 0:
            assert n_gpu == n_ref, f"seq {i}: num_accepted {n_gpu} != {n_ref}"
            assert got == want, f"seq {i}: tokens {got} != {want}"
            continue
        ties += 1
        if kind == 1:     # accept-level tie at `row`: rows before it exact, the rest valid
            assert row <= n_gpu <= K, f"seq {i}: gpu n {n_gpu} outside [{row}, {K}] (tie row)"
            assert got[:row] == want[:row], f"seq {i}: tokens before the tie row differ"
            if drafts is not None:
                p0 = r0 - i
                assert got[:n_gpu] == [int(t) for t in drafts[p0:p0 + n_gpu]], \
                    f"seq {i}: kept tokens are not the drafts"
            if V is not None:
                assert 0 <= got[n_gpu] < V, f"seq {i}: drawn token {got[n_gpu]} outside [0, V)"
            assert got[n_gpu + 1:] == [-1] * (K - n_gpu), f"seq {i}: tokens after the draw"
        else:             # draw-level tie: n and accepted drafts exact, token in the tie set
            assert n_gpu == n_ref, f"seq {i}: num_accepted {n_gpu} != {n_ref} (draw tie)"
            assert got[:n_ref] == want[:n_ref]
            alts = ref["tie_alts"][i]
            assert got[n_ref] in alts, f"seq {i}: drawn {got[n_ref]} not in tie set {alts}"
            assert got[n_ref + 1:] == [-1] * (K - n_ref)
    return B, ties


def tie_report(ref):
    """One line: sequences and positions inside the near-tie windows, by clause."""
    c = ref.get("tie_clauses", {})
    return (f"ties: {ref['tie_count']} sequences, {ref.get('tie_positions', 0)} positions "
            f"(accept {c.get('accept', 0)}, cdf {c.get('cdf', 0)}, nucleus {c.get('nucleus', 0)})")
