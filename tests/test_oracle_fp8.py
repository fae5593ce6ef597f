"""Pins of the oracle's 8-bit (E4M3) K/V reading.

* every one of the 256 codes decodes to the value torch's float8_e4m3fn gives
  (an implementation of the same format independent of the oracle);
* a few codes whose values follow from the format by hand (bias 7, 3 mantissa
  bits, subnormals at exponent 0, the largest finite 448, NaN at S.1111.111);
* attention over E4M3 K/V with per-tensor scales equals the oracle's attention
  over the same values stored as float32 (E4M3 values times a power-of-two
  scale are exact in float32), so the scales enter where the definition puts
  them: scores = scale * q . (k_code * k_scale), out = softmax . (v_code * v_scale).
"""
import numpy as np
import torch

import oracle
import workloads as W


def test_all_codes_match_torch_float8():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.to_f64(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_hand_values():
    v = oracle.to_f64(np.array([0x00, 0x80, 0x01, 0x07, 0x08, 0x38, 0x3C, 0x7E, 0xFE, 0x7F, 0xFF],
                               dtype=np.uint8))
    want = [0.0, -0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 1.5, 448.0, -448.0]
    assert list(v[:9]) == want
    assert np.isnan(v[9]) and np.isnan(v[10])


def test_fp8_attention_equals_float32_attention_of_the_same_values():
    w = W.workload("bass_b8", B=3, Hq=4, Hkv=2, D=64, L_lo=5, L_hi=90, K_lo=0, K_hi=4,
                   kv_dtype="e4m3", kv_scale=0.125, gen_seed=3)
    inp = W.make_inputs(w, with_logits=False)
    assert inp["k_cache"].dtype == np.uint8
    args = (inp["cu_q"], inp["kv_start"], inp["kv_len"], inp["num_kv_heads"])
    got = oracle.verify_attention(inp["q"], inp["k_new"], inp["v_new"], inp["k_cache"],
                                  inp["v_cache"], *args, k_scale=0.125, v_scale=0.125)
    f32 = {k: (oracle.to_f64(inp[k]) * 0.125).astype(np.float32)
           for k in ("k_new", "v_new", "k_cache", "v_cache")}
    assert all(np.array_equal(f32[k].astype(np.float64), oracle.to_f64(inp[k]) * 0.125)
               for k in f32)
    ref = oracle.verify_attention(inp["q"], f32["k_new"], f32["v_new"], f32["k_cache"],
                                  f32["v_cache"], *args)
    assert np.array_equal(got, ref)
    # and the scales matter: a different v_scale scales the output by the ratio
    got2 = oracle.verify_attention(inp["q"], inp["k_new"], inp["v_new"], inp["k_cache"],
                                   inp["v_cache"], *args, k_scale=0.125, v_scale=0.25)
    assert np.allclose(got2, 2 * got, rtol=1e-12, atol=0)


def test_e4m3_generation_round_trip():
    x = np.array([0.0, 1.0, -1.5, 0.3, 447.0, 1e-3], dtype=np.float32)
    c = W.f32_to_e4m3_codes(x)
    back = oracle.to_f64(c)
    assert back[0] == 0 and back[1] == 1 and back[2] == -1.5
    assert abs(back[3] - 0.3) <= 0.3 * 2 ** -4          # 3 mantissa bits: half an ulp
    assert back[4] == 448.0 and abs(back[5] - 1e-3) <= 2 ** -10
