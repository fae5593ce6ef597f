"""Sequence sharding across ranks, on CPU with two gloo ranks.

Each rank verifies its contiguous shard of one global batch (global sequence
ids kept) with the oracle; gathered in rank order, the results must equal the
single-process oracle on the whole batch, bit for bit: the step has no
exchange on the data path and its uniforms are keyed by global sequence id.
The max-over-ranks timing reduction of the benchmark is checked on the same
process group.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import workloads as W
from speculative_decoding_verify_09_gb300 import shard


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _batch(prefix=False):
    if prefix:
        w = W.workload("shared_prefix_s32", B=6, groups=3, prefix_lens=(40, 0, 25), Hq=2, Hkv=2,
                       D=64, V=300, L_lo=3, L_hi=30, K_lo=1, K_hi=4, gen_seed=77)
    else:
        w = W.workload("bass_b8", B=5, Hq=4, Hkv=2, D=64, V=300, L_lo=5, L_hi=60, K_lo=0,
                       K_hi=5, gen_seed=76, philox_seed=123)
    inp = W.make_inputs(w)
    inp["seq_ids"] = np.arange(inp["B"], dtype=np.int64) + 1000      # global ids
    return inp


def _flat(res, inp):
    """Per-sequence results of one oracle step, in sequence order."""
    cu = inp["cu_q"]
    rows = []
    for i in range(inp["B"]):
        a, b = int(cu[i]), int(cu[i + 1])
        start, L = int(inp["kv_start"][i]), int(inp["kv_len"][i])
        n = int(res["num_accepted"][i])
        app = res["k_cache"][start + L:start + L + max(n + 1, 0)]
        rows.append((n, res["out_tokens"][a:b].tolist(), res["out"][a:b].tobytes(),
                     int(res["new_kv_len"][i]), app.tobytes()))
    return rows


def _worker(rank, world, port, prefix, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = _batch(prefix)
        part = shard.shard_inputs(inp, rank, world)
        res = oracle.verify_step(part)
        mine = _flat(res, part)
        gathered = [None] * world
        dist.all_gather_object(gathered, mine)
        m = shard.max_over_ranks(1.5 + rank, dist)
        s = shard.sum_over_ranks(part["B"], dist)
        if rank == 0:
            q.put((sum(gathered, []), m, s))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("prefix", [False, True])
def test_two_gloo_ranks_equal_single_process(prefix):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, prefix, q)) for r in range(2)]
    for p in procs:
        p.start()
    got, m, s = q.get(timeout=300)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    inp = _batch(prefix)
    want = _flat(oracle.verify_step(inp), inp)
    assert got == want
    assert m == 2.5
    assert s == inp["B"]


def test_rank_ranges_cover_and_keep_groups():
    for B in (1, 5, 8, 33):
        for world in (1, 2, 3, 8):
            cuts = [shard.rank_range(B, r, world) for r in range(world)]
            assert cuts[0][0] == 0 and cuts[-1][1] == B
            assert all(cuts[r][1] == cuts[r + 1][0] for r in range(world - 1))
    group = np.array([0, 0, 0, 1, 1, 2, 2, 2, 2])
    for world in (2, 3, 4):
        for r in range(world):
            lo, hi = shard.rank_range(len(group), r, world, group)
            if 0 < lo < len(group):
                assert group[lo] != group[lo - 1]
