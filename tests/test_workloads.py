"""The seeded input generator: reproducible, shaped as declared."""
import numpy as np

import workloads as W


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1e-3], dtype=np.float32)
    b = W.f32_to_bf16_bits(x)
    back = W.bf16_bits_to_f32(b)
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == 1.0 + 2 ** -6
    assert back[3] == -2.5 and abs(back[4] - 1e-3) / 1e-3 < 2 ** -8


def test_reproducible_and_shaped():
    w = W.workload("ragged_gqa_b32", B=5, V=300, L_hi=200)
    a, b = W.make_inputs(w), W.make_inputs(w)
    for k in ("q", "k_cache", "target_logits", "draft_tokens", "kv_len", "cu_q"):
        assert np.array_equal(a[k], b[k])
    R = int(a["cu_q"][-1])
    assert a["q"].shape == (R, 32, 128) and a["k_new"].shape == (R, 8, 128)
    assert a["target_logits"].shape == (R, 300) and a["draft_logits"].shape == (R - 5, 300)
    K = np.diff(a["cu_q"]) - 1
    assert np.all((K >= 1) & (K <= 8))
    assert np.all(a["kv_cap"] >= a["kv_len"] + K + 1)
    assert np.all(a["kv_start"][1:] >= a["kv_start"][:-1] + a["kv_cap"][:-1])
    assert a["kv_start"][-1] + a["kv_cap"][-1] <= a["pool_rows"]
    assert np.all((a["draft_tokens"] >= 0) & (a["draft_tokens"] < 300))


def test_shared_prefix_layout():
    a = W.make_inputs(W.workload("shared_prefix_s32", B=4, V=64, prefix_len=100),
                      with_logits=False)
    assert a["prefix_start"][0] + a["prefix_len"][0] <= a["kv_start"][0]
    assert np.all(a["group"] == 0)


def test_step_bytes_bass_shape():
    a = W.make_inputs(W.workload("bass_b8"), with_attention=False, with_logits=False)
    nb = W.step_bytes(a)
    assert nb["attention"] > 8 * 512 * 32 * 128 * 4


def test_step_bytes_count_every_tensor_once():
    """Algorithmic bytes written out by hand for a small batch: the KV rows
    read once, the block's q, out and new K/V, every logits row, and the
    append's read + write of all block rows; an E4M3 cache counts one byte
    per K/V element and leaves q, out and the logits unchanged."""
    w = W.workload("bass_b8", B=3, Hq=4, Hkv=2, D=64, V=100, L_lo=10, L_hi=30, K_lo=2, K_hi=2,
                   gen_seed=9)
    a = W.make_inputs(w, with_attention=False, with_logits=False)
    L = int(np.sum(a["kv_len"]))
    R = 9                                           # 3 sequences x (K + 1)
    kv = L * 2 * 64 * 2 * 2                         # K and V cache rows, bf16
    block = R * (2 * 4 * 64 * 2 + 2 * 2 * 64 * 2)   # q + out, k_new + v_new
    nb = W.step_bytes(a)
    assert nb["attention"] == kv + block
    assert nb["sampler"] == (2 * R - 3) * 100 * 2
    assert nb["append"] == 2 * R * 2 * 64 * 2 * 2
    a8 = dict(a, kv_dtype="e4m3")
    nb8 = W.step_bytes(a8)
    assert nb8["attention"] == kv // 2 + R * 2 * 4 * 64 * 2 + R * 2 * 2 * 64
    assert nb8["sampler"] == nb["sampler"] and nb8["append"] == nb["append"] // 2


def test_draft_inputs_positions_and_bytes():
    w = W.workload("bass_b8", B=4, Hq=4, Hkv=4, D=64, V=50, L_lo=5, L_hi=20, gen_seed=3)
    base, steps = W.make_draft_inputs(w, positions=3)
    assert list(base["cu_q"]) == [0, 1, 2, 3, 4]
    assert np.all(base["kv_cap"] == base["kv_len"] + 3)       # room for three positions
    assert all(st["q"].shape == (4, 4, 64) and st["draft_logits"].shape == (4, 50)
               for st in steps)
    assert not np.array_equal(steps[0]["q"], steps[1]["q"])
    L = int(np.sum(base["kv_len"]))
    assert W.draft_step_bytes(base) == (L * 4 * 64 * 2 * 2 + 4 * (2 * 4 + 2 * 4) * 64 * 2
                                        + 4 * 50 * 2 + 2 * 4 * 2 * 4 * 64 * 2)


def test_padded_step_bytes_by_hand():
    """Padding every cache to the longest and every block to the largest K:
    written out for three sequences."""
    w = W.workload("bass_b8", B=3, Hq=4, Hkv=2, D=64, V=100, L_dist="fixed",
                   L_fixed=(10, 40, 25), K_fixed=(1, 4, 2), gen_seed=5)
    a = W.make_inputs(w, with_attention=False, with_logits=False)
    nb = W.padded_step_bytes(a)
    assert nb["attention"] == 3 * 40 * 2 * 64 * 2 * 2 + 3 * 5 * (2 * 4 + 2 * 2) * 64 * 2
    assert nb["sampler"] == (2 * 15 - 3) * 100 * 2
    assert nb["append"] == 2 * 15 * 2 * 64 * 2 * 2
    flat = W.step_bytes(a)
    assert flat["attention"] == 75 * 2 * 64 * 2 * 2 + 10 * (2 * 4 + 2 * 2) * 64 * 2
    assert nb["total"] > flat["total"]
