"""Pins of the oracle's verify attention.

Sources: "Accelerating Large Language Model Decoding with Speculative
Sampling", section "Conditional scoring" (K+1 rows scored in one call over the
KV cache); BASS / EMS-SD abstracts (ragged batch, no padding); bifurcated
attention abstract (prefix + decode split is precise: equal to attention over
the concatenated KV).
"""
import math

import numpy as np
import pytest

from oracle.attention import attention_row, verify_attention
import workloads as W


def _rand_case(seed, B=3, Hq=4, Hkv=2, D=8, Ls=(0, 5, 11), Rs=(1, 3, 4)):
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(Rs)]).astype(np.int32)
    R = int(cu[-1])
    starts = np.concatenate([[2], 2 + np.cumsum(np.array(Ls) + 6)[:-1]]).astype(np.int64)
    P = int(starts[-1] + Ls[-1] + 8)
    f = lambda *s: rng.normal(size=s).astype(np.float32)
    return dict(q=f(R, Hq, D), k_new=f(R, Hkv, D), v_new=f(R, Hkv, D), k_cache=f(P, Hkv, D),
                v_cache=f(P, Hkv, D), cu_q=cu, kv_start=starts,
                kv_len=np.array(Ls, dtype=np.int32), num_kv_heads=Hkv)


def _call(c, **kw):
    return verify_attention(c["q"], c["k_new"], c["v_new"], c["k_cache"], c["v_cache"],
                            c["cu_q"], c["kv_start"], c["kv_len"], c["num_kv_heads"], **kw)


def test_matches_pure_python_loops():
    """Independent scalar formulation: explicit loops, math.exp, no matmul."""
    c = _rand_case(0)
    out = _call(c)
    Hq, Hkv, D = 4, 2, 8
    g = Hq // Hkv
    for i in range(3):
        L, a, r0 = int(c["kv_len"][i]), int(c["kv_start"][i]), int(c["cu_q"][i])
        for j in range(int(c["cu_q"][i + 1]) - r0):
            for h in range(Hq):
                hk = h // g
                keys = [c["k_cache"][a + t, hk] for t in range(L)] + \
                       [c["k_new"][r0 + b, hk] for b in range(j + 1)]
                vals = [c["v_cache"][a + t, hk] for t in range(L)] + \
                       [c["v_new"][r0 + b, hk] for b in range(j + 1)]
                sc = float(np.float32(1 / math.sqrt(D)))
                s = [sc * sum(float(c["q"][r0 + j, h, d]) * float(k[d]) for d in range(D))
                     for k in keys]
                m = max(s)
                e = [math.exp(x - m) for x in s]
                z = sum(e)
                for d in range(D):
                    want = sum(e[t] * float(vals[t][d]) for t in range(len(e))) / z
                    assert abs(out[r0 + j, h, d] - want) < 1e-12


def test_single_visible_key_returns_its_value():
    c = _rand_case(1, B=1, Ls=(0,), Rs=(3,))
    out = _call(c)
    for h in range(4):
        assert np.array_equal(out[0, h], c["v_new"][0, h // 2].astype(np.float64))


def test_zero_query_gives_mean_of_visible_values():
    c = _rand_case(2)
    c["q"][:] = 0
    out = _call(c)
    i, j, h = 2, 2, 3
    r0, a, L = int(c["cu_q"][i]), int(c["kv_start"][i]), int(c["kv_len"][i])
    vis = np.concatenate([c["v_cache"][a:a + L, h // 2], c["v_new"][r0:r0 + j + 1, h // 2]])
    assert np.allclose(out[r0 + j, h], vis.astype(np.float64).mean(0), atol=1e-14)


def test_causal_block_future_rows_have_no_effect():
    c = _rand_case(3)
    out = _call(c)
    i = 2
    r0 = int(c["cu_q"][i])
    c["k_new"][r0 + 2:r0 + 4] += 5.0
    c["v_new"][r0 + 2:r0 + 4] -= 3.0
    out2 = _call(c)
    assert np.array_equal(out[r0:r0 + 2], out2[r0:r0 + 2])
    assert not np.allclose(out[r0 + 2], out2[r0 + 2])


def test_batch_equals_each_sequence_alone():
    c = _rand_case(4)
    out = _call(c)
    for i in range(3):
        r0, r1 = int(c["cu_q"][i]), int(c["cu_q"][i + 1])
        one = verify_attention(c["q"][r0:r1], c["k_new"][r0:r1], c["v_new"][r0:r1],
                               c["k_cache"], c["v_cache"], np.array([0, r1 - r0]),
                               c["kv_start"][i:i + 1], c["kv_len"][i:i + 1], 2)
        assert np.array_equal(one, out[r0:r1])


def test_shared_prefix_equals_concatenated_cache():
    """Bifurcated mode == plain attention with the prefix copied in front of
    each sequence's own rows."""
    rng = np.random.default_rng(5)
    Hq = Hkv = 2
    D, Pl = 8, 13
    Ls, Rs = [0, 4, 9], [2, 3, 1]
    B = 3
    cu = np.concatenate([[0], np.cumsum(Rs)]).astype(np.int32)
    R = int(cu[-1])
    f = lambda *s: rng.normal(size=s).astype(np.float32)
    pool = f(64, Hkv, D), f(64, Hkv, D)
    starts = np.array([20, 30, 40], dtype=np.int64)
    q, kn, vn = f(R, Hq, D), f(R, Hkv, D), f(R, Hkv, D)
    bif = verify_attention(q, kn, vn, pool[0], pool[1], cu, starts, np.array(Ls), Hkv,
                           prefix=(np.zeros(B, np.int32), np.array([3]), np.array([Pl])))
    # concatenated layout: each sequence gets prefix ++ own rows, contiguous
    k2, v2 = np.zeros((200, Hkv, D), np.float32), np.zeros((200, Hkv, D), np.float32)
    st2 = np.array([0, 60, 120], dtype=np.int64)
    for i in range(B):
        for src, dst in ((pool[0], k2), (pool[1], v2)):
            dst[st2[i]:st2[i] + Pl] = src[3:3 + Pl]
            dst[st2[i] + Pl:st2[i] + Pl + Ls[i]] = src[starts[i]:starts[i] + Ls[i]]
    cat = verify_attention(q, kn, vn, k2, v2, cu, st2, np.array(Ls) + Pl, Hkv)
    assert np.allclose(bif, cat, atol=1e-13, rtol=0)


def test_bf16_inputs_are_read_exactly():
    c = _rand_case(6)
    bf = {k: (W.f32_to_bf16_bits(v) if isinstance(v, np.ndarray) and v.dtype == np.float32
              else v) for k, v in c.items()}
    f32 = {k: (W.bf16_bits_to_f32(v) if isinstance(v, np.ndarray) and v.dtype == np.uint16
               else v) for k, v in bf.items()}
    assert np.array_equal(_call(bf), _call(f32))


def test_explicit_scale():
    c = _rand_case(7)
    a = _call(c, scale=0.5)
    c2 = dict(c)
    c2["q"] = c["q"] * np.float32(0.5 * math.sqrt(8))
    b = _call(c2)
    assert np.allclose(a, b, atol=1e-12)
