"""Philox4x32-10 counter-based generator and the verify step's uniforms.

TEST INFRASTRUCTURE ONLY: this module belongs to the CPU oracle.  Only tests,
the smoke check and the bench's CPU-baseline leg may import it.

Source of the generator: Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers:
As Easy as 1, 2, 3" (SC'11), section "Philox".  A Philox4x32 round multiplies
counter words 0 and 2 by two fixed 32-bit constants, keeps the high and low
halves of both 64-bit products, and mixes the high halves into words 1 and 3
with the round key; the 2-word key is advanced by two Weyl constants between
rounds.  Ten rounds are used (the "-10" variant the paper recommends).

Use in the method: "Accelerating Large Language Model Decoding with
Speculative Sampling" (Chen et al.), section "Modified rejection sampling",
needs one uniform per acceptance test and one per (re)sampling draw; the page
fixes no generator (its results section only notes that seeding differs from
plain sampling).  Reading taken here: the counter is (position, low32(seq_id),
high32(seq_id), stream), the key is (low32(seed), high32(seed)); word 0 gives
the acceptance uniform and word 1 the sampling uniform, each as
u = (w >> 8) * 2^-24, a 24-bit value exact in fp32 and fp64.

Pins: the known-answer vectors published with the generator's reference
implementation (Random123: counter and key all zero, all ones, and the
pi-digit counter/key) are matched exactly; the tests also pin invertibility of
the rounds, the constants, and the statistical properties the method needs.
"""
import numpy as np

# Multipliers and Weyl key increments of Philox4x32 (SC'11, section "Philox").
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
ROUNDS = 10

STREAM_VERIFY = 0   # uniforms consumed by the verify step
STREAM_DRAFT = 1    # reserved for drawing draft tokens (never used by verify)

_MASK32 = np.uint64(0xFFFFFFFF)


def _u64(x):
    return np.asarray(x, dtype=np.uint64) & _MASK32


def philox4x32(c0, c1, c2, c3, k0, k1, rounds=ROUNDS):
    """Apply `rounds` Philox4x32 rounds to counter (c0..c3) under key (k0, k1).

    All arguments broadcast (numpy arrays or ints, values < 2**32); returns four
    uint64 arrays holding 32-bit words.
    """
    c0, c1, c2, c3 = _u64(c0), _u64(c1), _u64(c2), _u64(c3)
    k0, k1 = _u64(k0), _u64(k1)
    m0, m1 = np.uint64(PHILOX_M0), np.uint64(PHILOX_M1)
    for r in range(rounds):
        if r > 0:
            k0 = (k0 + np.uint64(PHILOX_W0)) & _MASK32
            k1 = (k1 + np.uint64(PHILOX_W1)) & _MASK32
        p0 = m0 * c0          # < 2**64: product of two 32-bit values
        p1 = m1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c0, c1, c2, c3 = (hi1 ^ c1 ^ k0), lo1, (hi0 ^ c3 ^ k1), lo0
    return c0, c1, c2, c3


def word_to_uniform(w):
    """Top 24 bits of a 32-bit word as a float64 in [0, 1): (w >> 8) * 2^-24."""
    return (_u64(w) >> np.uint64(8)).astype(np.float64) * (2.0 ** -24)


def verify_uniforms(seed, seq_id, pos, stream=STREAM_VERIFY):
    """(u_acc, u_smp) for the decision at absolute token index `pos` of `seq_id`.

    seed: uint64; seq_id: int64 (two's complement bits are used); pos: uint32.
    Broadcasts over array arguments.
    """
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    sid = np.asarray(seq_id, dtype=np.int64).astype(np.uint64)
    w0, w1, _, _ = philox4x32(pos, sid & _MASK32, sid >> np.uint64(32), stream,
                              seed & 0xFFFFFFFF, seed >> 32)
    return word_to_uniform(w0), word_to_uniform(w1)
