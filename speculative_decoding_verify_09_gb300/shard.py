"""Sequence sharding of a verify batch across ranks (one GPU per rank).

Sequences are independent units of the verify step: the attention, the
decisions and the append of sequence i touch only sequence i's rows, and the
uniforms are keyed by the global sequence id (Philox counter (position,
seq_id)), so a batch split into contiguous sequence ranges gives the same
results on any number of ranks with no exchange on the data path.  Groups
sharing a prefix stay on one rank.  This module holds the host-side logic:
which sequences a rank owns, its sub-batch of a host input dict, and the
max-over-ranks reduction the benchmark uses for timing.
"""
import numpy as np


def rank_range(num_seqs, rank, world, group=None):
    """Contiguous sequence range [lo, hi) of `rank` among `world` ranks.

    Balanced by count; with `group` ([B] non-decreasing group ids) the cut
    points move forward to the next group start so no group is split."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside world of {world}")

    def cut(r):
        c = (num_seqs * r) // world
        if group is not None and 0 < c < num_seqs:
            while c < num_seqs and group[c] == group[c - 1]:
                c += 1
        return c

    return cut(rank), cut(rank + 1)


_ROW_KEYS = ("q", "k_new", "v_new", "target_logits")
_DRAFT_KEYS = ("draft_logits", "draft_tokens")
_SEQ_KEYS = ("kv_start", "kv_len", "kv_cap")


def shard_inputs(inp, rank, world):
    """The sub-batch of host input dict `inp` owned by `rank`.

    Block rows, logits rows and draft rows are sliced to the rank's sequences,
    cu_q is rebased, per-sequence arrays are sliced and seq_ids keep their
    global values.  KV pools (and shared prefixes) are shared, not copied: the
    rank's sequences address their own rows through kv_start."""
    B = int(inp["B"])
    lo, hi = rank_range(B, rank, world, inp.get("group"))
    cu = np.asarray(inp["cu_q"])
    r0, r1 = int(cu[lo]), int(cu[hi])
    d0, d1 = r0 - lo, r1 - hi
    out = dict(inp)
    out["B"] = hi - lo
    out["cu_q"] = (cu[lo:hi + 1] - r0).astype(cu.dtype)
    seq_ids = inp.get("seq_ids")
    out["seq_ids"] = (np.arange(B, dtype=np.int64) if seq_ids is None else np.asarray(seq_ids))[lo:hi].copy()
    for k in _ROW_KEYS:
        if inp.get(k) is not None:
            out[k] = inp[k][r0:r1]
    for k in _DRAFT_KEYS:
        if inp.get(k) is not None:
            out[k] = inp[k][d0:d1]
    for k in _SEQ_KEYS:
        if inp.get(k) is not None:
            out[k] = inp[k][lo:hi]
    if inp.get("group") is not None:
        g = np.asarray(inp["group"])[lo:hi]
        g0 = int(g[0]) if len(g) else 0
        g1 = int(g[-1]) + 1 if len(g) else 0
        out["group"] = (g - g0).astype(g.dtype)
        out["prefix_start"] = inp["prefix_start"][g0:g1]
        out["prefix_len"] = inp["prefix_len"][g0:g1]
    out["shard"] = (lo, hi, r0, r1)
    return out


def max_over_ranks(value, dist=None, device=None):
    """max of a float over all ranks (the value itself without a process group)."""
    if dist is None or not dist.is_available() or not dist.is_initialized():
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value, dist=None, device=None):
    """sum of a number over all ranks (the value itself without a process group)."""
    if dist is None or not dist.is_available() or not dist.is_initialized():
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t)
    return t.item()
