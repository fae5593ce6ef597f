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
