"""Pins of the oracle's ragged append (EMS-SD abstract: each sample keeps its
own accepted count, no padding, no extra memory)."""
import numpy as np

from oracle.append import kv_append
from oracle.sampling import DEV_CAPACITY


def test_append_rows_lengths_and_untouched_rows():
    rng = np.random.default_rng(0)
    Hkv, D = 2, 4
    Ls = np.array([3, 0, 5], dtype=np.int32)
    Rs = [4, 2, 3]
    cu = np.concatenate([[0], np.cumsum(Rs)]).astype(np.int32)
    starts = np.array([1, 10, 20], dtype=np.int64)
    cap = np.array([7, 2, 6], dtype=np.int32)
    kc = rng.normal(size=(30, Hkv, D)).astype(np.float32)
    vc = rng.normal(size=(30, Hkv, D)).astype(np.float32)
    kn = rng.normal(size=(9, Hkv, D)).astype(np.float32)
    vn = rng.normal(size=(9, Hkv, D)).astype(np.float32)
    nacc = np.array([2, 1, 2], dtype=np.int32)       # seq 2: 5 + 3 > 6 -> overflow
    k2, v2, nl, st = kv_append(kc, vc, kn, vn, cu, starts, Ls, cap, nacc)
    assert list(nl) == [6, 2, 5] and st == DEV_CAPACITY
    expect_k, expect_v = kc.copy(), vc.copy()
    expect_k[4:7], expect_v[4:7] = kn[0:3], vn[0:3]
    expect_k[10:12], expect_v[10:12] = kn[4:6], vn[4:6]
    assert np.array_equal(k2, expect_k) and np.array_equal(v2, expect_v)


def test_failed_sequence_is_not_appended():
    kc = np.zeros((8, 1, 2), np.float32)
    kn = np.ones((2, 1, 2), np.float32)
    k2, v2, nl, st = kv_append(kc, kc, kn, kn, np.array([0, 2]), np.array([0]),
                               np.array([3]), np.array([8]), np.array([-1]))
    assert list(nl) == [3] and st == 0 and not k2.any()
