"""Seeded synthetic inputs for the verify step (shared by the oracle's tests,
the CUDA path's tests and the bench).

This module holds none of the verify step's arithmetic: it only draws random
tensors with numpy's PCG64 and lays them out.  Workload shapes follow the
pages' setting -- 7-8B-class attention shapes, batch 8-64, 4-8 drafts, 32000 or
128256 vocabularies (BASS abstract: 7.8B model at batch 8; speculative
sampling, section "Experimental setup": K = 4, nucleus 0.8 / 0.95,
temperature 0.8; bifurcated attention abstract: 32 samples over an 8k shared
context).  The evaluation datasets the pages use are not available; these
draws stand in for them.

Layouts (all host numpy arrays):
  q [R, Hq, D], k_new / v_new [R, Hkv, D]        block rows of every sequence
  k_cache / v_cache [P, Hkv, D]                  token-major KV pool
  cu_q [B+1] int32, kv_start [B] int64, kv_len [B] int32, kv_cap [B] int32
  target_logits [R, V], draft_logits [R-B, V], draft_tokens [R-B] int32
  seq_ids [B] int64; group [B] int32, prefix_start [G] int64, prefix_len [G]
  int32 (shared-prefix mode only)
Float tensors are float32 arrays, or bfloat16 stored as uint16 bit patterns
(rounded to nearest even from float32 draws).  With kv_dtype "e4m3" the K/V
tensors (cache and block rows) are E4M3 codes (uint8) of float32 N(0, 1)
draws divided by kv_scale, rounded to nearest even; the input dict then also
holds kv_dtype, k_scale and v_scale.

Draft tokens are drawn from softmax(draft_logits / T) over the full vocabulary
(Gumbel-max with this module's RNG; the row's argmax when T = 0), standing in
for the draft model's own sampler.
"""
from dataclasses import dataclass, replace
import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    dtype: str                 # "f32" | "bf16"
    V: int
    L_lo: int                  # committed KV rows per sequence, lower bound
    L_hi: int                  # ... upper bound (inclusive)
    L_dist: str = "uniform"    # "uniform" | "loguniform" | "fixed"
    L_fixed: tuple = ()
    K_lo: int = 4              # drafts per sequence, lower bound
    K_hi: int = 4              # ... upper bound (inclusive)
    K_fixed: tuple = ()        # explicit per-sequence draft counts (overrides K_lo/K_hi)
    logit_std: float = 3.0
    draft_noise: float = 1.0
    temperature: float = 1.0
    top_p: float = 1.0
    top_k: int = 0             # 0: no top-k
    philox_seed: int = 0
    prefix_len: int = 0        # > 0: shared prefixes of this length (bifurcated)
    groups: int = 1            # shared-prefix groups (contiguous runs of sequences)
    prefix_lens: tuple = ()    # per-group prefix lengths (overrides prefix_len)
    cap_slack: int = 0         # extra pool rows per sequence beyond L + K + 1
    gen_seed: int = 0
    kv_dtype: str = ""         # "" (same as dtype) | "e4m3": 8-bit K/V codes
    kv_scale: float = 0.0625   # per-tensor K/V scale of an e4m3 cache (code value x scale)


# The five workloads (sizes as the pages' setting suggests; see module doc).
WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", B=2, Hq=4, Hkv=4, D=64, dtype="f32", V=256,
                         L_lo=17, L_hi=40, L_dist="fixed", L_fixed=(17, 40),
                         K_lo=4, K_hi=4, logit_std=2.0, draft_noise=0.5, gen_seed=1),
    "bass_b8": Workload("bass_b8", B=8, Hq=32, Hkv=32, D=128, dtype="bf16", V=32000,
                        L_lo=512, L_hi=2048, K_lo=5, K_hi=5, logit_std=3.0,
                        draft_noise=1.0, gen_seed=2),
    "ragged_gqa_b32": Workload("ragged_gqa_b32", B=32, Hq=32, Hkv=8, D=128, dtype="bf16",
                               V=32000, L_lo=128, L_hi=8192, L_dist="loguniform",
                               K_lo=1, K_hi=8, logit_std=3.0, draft_noise=1.0,
                               temperature=0.8, top_p=0.95, gen_seed=3),
    "shared_prefix_s32": Workload("shared_prefix_s32", B=32, Hq=32, Hkv=32, D=128,
                                  dtype="bf16", V=32000, L_lo=0, L_hi=512, K_lo=4,
                                  K_hi=4, logit_std=3.0, draft_noise=1.0,
                                  prefix_len=8192, gen_seed=4),
    "vocab128k_b64": Workload("vocab128k_b64", B=64, Hq=32, Hkv=8, D=128, dtype="bf16",
                              V=128256, L_lo=1024, L_hi=4096, K_lo=8, K_hi=8,
                              logit_std=4.0, draft_noise=1.0, temperature=0.7,
                              top_p=0.9, gen_seed=5),
}


def workload(name, **overrides):
    w = WORKLOADS[name]
    return replace(w, **overrides) if overrides else w


def f32_to_bf16_bits(x):
    """float32 -> bfloat16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits):
    """bfloat16 bit patterns -> float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal(rng, shape, std, dtype):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return f32_to_bf16_bits(x) if dtype == "bf16" else x


def f32_to_e4m3_codes(x):
    """float32 -> E4M3 codes (uint8), round to nearest even, by torch's
    float8_e4m3fn conversion (finite inputs within +-448)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _kv(rng, shape, w):
    """K or V rows: N(0, 1) draws, stored as the workload's K/V type."""
    if w.kv_dtype == "e4m3":
        x = rng.standard_normal(size=shape, dtype=np.float32)
        return f32_to_e4m3_codes(x / np.float32(w.kv_scale))
    return _normal(rng, shape, 1.0, w.dtype)


def _as_f32(x):
    return bf16_bits_to_f32(x) if x.dtype == np.uint16 else x


def draw_lengths(w, rng):
    if w.L_dist == "fixed":
        L = np.array(w.L_fixed, dtype=np.int64)
    elif w.L_dist == "loguniform":
        L = np.rint(np.exp(rng.uniform(np.log(w.L_lo), np.log(w.L_hi), size=w.B)))
    else:
        L = rng.integers(w.L_lo, w.L_hi + 1, size=w.B)
    K = rng.integers(w.K_lo, w.K_hi + 1, size=w.B)
    if w.K_fixed:
        K = np.array(w.K_fixed, dtype=np.int64)
    return L.astype(np.int64), K.astype(np.int64)


def make_inputs(w, with_attention=True, with_logits=True, guard_rows=8):
    """Draw one step's inputs for workload `w` (a Workload)."""
    rng = np.random.Generator(np.random.PCG64(w.gen_seed))
    L, K = draw_lengths(w, rng)
    R_i = K + 1
    cu_q = np.zeros(w.B + 1, dtype=np.int32)
    cu_q[1:] = np.cumsum(R_i)
    R = int(cu_q[-1])
    cap = L + R_i + w.cap_slack
    # pool: guard | prefixes | seq0 region | seq1 region | ... | guard
    prefix_start = None
    base = guard_rows
    shared = w.prefix_len > 0 or len(w.prefix_lens) > 0
    if shared:
        plen = np.array(w.prefix_lens if w.prefix_lens else [w.prefix_len] * w.groups,
                        dtype=np.int64)
        prefix_start = base + np.concatenate([[0], np.cumsum(plen)[:-1]]).astype(np.int64)
        base += int(plen.sum())
    kv_start = np.zeros(w.B, dtype=np.int64)
    kv_start[0] = base
    kv_start[1:] = base + np.cumsum(cap)[:-1]
    P = int(base + cap.sum() + guard_rows)
    inp = dict(workload=w, B=w.B, V=w.V, num_q_heads=w.Hq, num_kv_heads=w.Hkv,
               head_dim=w.D, dtype=w.dtype, cu_q=cu_q, kv_start=kv_start,
               kv_len=L.astype(np.int32), kv_cap=cap.astype(np.int32),
               seq_ids=np.arange(w.B, dtype=np.int64),
               temperature=w.temperature, top_p=w.top_p, top_k=w.top_k, seed=w.philox_seed,
               scale=0.0, pool_rows=P)
    if shared:
        G = len(plen)
        inp.update(group=(np.arange(w.B) * G // w.B).astype(np.int32), prefix_start=prefix_start,
                   prefix_len=plen.astype(np.int32))
    if with_attention:
        inp["q"] = _normal(rng, (R, w.Hq, w.D), 1.0, w.dtype)
        inp["k_new"] = _kv(rng, (R, w.Hkv, w.D), w)
        inp["v_new"] = _kv(rng, (R, w.Hkv, w.D), w)
        inp["k_cache"] = _kv(rng, (P, w.Hkv, w.D), w)
        inp["v_cache"] = _kv(rng, (P, w.Hkv, w.D), w)
        if w.kv_dtype == "e4m3":
            inp.update(kv_dtype="e4m3", k_scale=w.kv_scale, v_scale=w.kv_scale)
    if with_logits:
        tgt = rng.standard_normal(size=(R, w.V), dtype=np.float32) * np.float32(w.logit_std)
        # draft row j of sequence i sits next to target row j of the same sequence
        src = np.concatenate([np.arange(cu_q[i], cu_q[i + 1] - 1) for i in range(w.B)])
        drf = tgt[src] + rng.standard_normal(size=(R - w.B, w.V),
                                             dtype=np.float32) * np.float32(w.draft_noise)
        if w.dtype == "bf16":
            tgt, drf = f32_to_bf16_bits(tgt), f32_to_bf16_bits(drf)
        inp["target_logits"], inp["draft_logits"] = tgt, drf
        # stand-in draft sampler: Gumbel-max on draft_logits / T, row by row
        toks = np.empty(R - w.B, dtype=np.int32)
        for r in range(R - w.B):
            if w.temperature == 0.0:         # greedy drafting: the draft row's argmax
                toks[r] = int(np.argmax(_as_f32(drf[r])))
                continue
            g = -np.log(-np.log(rng.uniform(np.finfo(np.float32).tiny, 1.0,
                                            size=w.V).astype(np.float64)))
            toks[r] = int(np.argmax(_as_f32(drf[r]).astype(np.float64) / w.temperature + g))
        inp["draft_tokens"] = toks
    return inp


def make_draft_inputs(w, positions=1):
    """Inputs of `positions` consecutive draft positions for workload `w`.

    Each position is one decode step of the draft model: one block row per
    sequence (cu_q = 0..B).  The cache is laid out as in make_inputs (drawn
    with K_i = 0) with room for `positions` more rows per sequence.  Returns
    (base, steps): base is the input dict of position 0 with its
    `draft_logits` [B, V] (standing in for the draft model's outputs); steps[t]
    holds position t's q [B, Hq, D], k_new / v_new [B, Hkv, D] and
    draft_logits, position 0's equal to base's, later ones drawn afresh.
    """
    wd = replace(w, K_fixed=(0,) * w.B, cap_slack=w.cap_slack + positions - 1)
    base = make_inputs(wd)
    base["draft_logits"] = base.pop("target_logits")
    base.pop("draft_tokens", None)
    steps = [{k: base[k] for k in ("q", "k_new", "v_new", "draft_logits")}]
    for t in range(1, positions):
        rng = np.random.Generator(np.random.PCG64([w.gen_seed, t]))
        st = {"q": _normal(rng, (w.B, w.Hq, w.D), 1.0, w.dtype),
              "k_new": _kv(rng, (w.B, w.Hkv, w.D), w),
              "v_new": _kv(rng, (w.B, w.Hkv, w.D), w)}
        lg = rng.standard_normal(size=(w.B, w.V), dtype=np.float32) * np.float32(w.logit_std)
        st["draft_logits"] = f32_to_bf16_bits(lg) if w.dtype == "bf16" else lg
        steps.append(st)
    return base, steps


def draft_step_bytes(inp):
    """Algorithmic HBM bytes of one draft position on these inputs: the KV
    rows read once, q, the new K/V row and the output, the draft logits rows,
    and the append's read + write of one row per sequence."""
    esz = 4 if inp["dtype"] == "f32" else 2
    Hq, Hkv, D, B = inp["num_q_heads"], inp["num_kv_heads"], inp["head_dim"], inp["B"]
    kv_rows = int(np.sum(inp["kv_len"]))
    attn = kv_rows * Hkv * D * esz * 2 + B * (2 * Hq + 2 * Hkv) * D * esz
    return attn + B * inp["V"] * esz + 2 * B * 2 * Hkv * D * esz


def padded_step_bytes(inp):
    """Bytes the same verify step would move with padding (the vanilla
    multi-sample method of the EMS-SD abstract): every sequence's cache read
    to the batch's longest, every block and logits range to the largest draft
    count, and the append of the longest block for every sequence.  Returned
    like step_bytes, for comparison with it; no kernel runs this way."""
    esz = 4 if inp["dtype"] == "f32" else 2
    kvsz = 1 if inp.get("kv_dtype") == "e4m3" else esz
    Hq, Hkv, D, B = inp["num_q_heads"], inp["num_kv_heads"], inp["head_dim"], inp["B"]
    Lmax = int(np.max(inp["kv_len"])) if B else 0
    Rmax = int(np.max(np.diff(inp["cu_q"]))) if B else 0
    kv_rows = B * Lmax
    if inp.get("group") is not None:
        kv_rows += int(np.sum(inp["prefix_len"]))
    R = B * Rmax
    attn = kv_rows * Hkv * D * kvsz * 2 + R * 2 * Hq * D * esz + R * 2 * Hkv * D * kvsz
    logits = (2 * R - B) * inp["V"] * esz
    append = 2 * R * Hkv * D * kvsz * 2
    return dict(attention=attn, sampler=logits, append=append, total=attn + logits + append)


def step_bytes(inp):
    """Algorithmic HBM bytes of one verify step on these inputs.

    KV rows read once (a shared prefix once per group), the block's Q, new K/V
    and the output, every target and draft logits row read once, and the
    append's read + write of the committed rows (counted for all K_i + 1 rows,
    an upper bound on n_i + 1).
    """
    esz = 4 if inp["dtype"] == "f32" else 2
    kvsz = 1 if inp.get("kv_dtype") == "e4m3" else esz
    Hq, Hkv, D = inp["num_q_heads"], inp["num_kv_heads"], inp["head_dim"]
    R = int(inp["cu_q"][-1])
    B = inp["B"]
    kv_rows = int(np.sum(inp["kv_len"]))
    if inp.get("group") is not None:
        kv_rows += int(np.sum(inp["prefix_len"]))
    attn = kv_rows * Hkv * D * kvsz * 2 + R * 2 * Hq * D * esz + R * 2 * Hkv * D * kvsz
    logits = (2 * R - B) * inp["V"] * esz
    append = 2 * R * Hkv * D * kvsz * 2
    return dict(attention=attn, sampler=logits, append=append,
                total=attn + logits + append)
