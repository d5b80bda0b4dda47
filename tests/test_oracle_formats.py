"""Pins of the oracle's number formats against library routines and published
tables (no GPU)."""
import os

import numpy as np
import pytest
import torch

import oracle as orc
from conftest import GOLDEN


def _golden_values():
    rows = []
    with open(os.path.join(GOLDEN, "fp4_fp8_values.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            fmt, code, val = line.split()
            rows.append((fmt, int(code, 16), float(val)))
    return rows


def test_bf16_rounding_matches_torch_on_f32_inputs():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),      # f32 subnormals
        (rng.standard_normal(2000) * 1e37).astype(np.float32),
        np.array([0.0, -0.0, 1.0, 3.3895314e38, 3.39e38, 3.4e38, 1e-45], np.float32),
    ])
    want = torch.from_numpy(vals).to(torch.bfloat16).to(torch.float64).numpy()
    got = orc.round_to_bf16(vals.astype(np.float64))
    np.testing.assert_array_equal(got, want)
    bits = orc.f64_to_bf16_bits(vals.astype(np.float64))
    want_bits = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(bits, want_bits)


def test_bf16_ties_and_single_rounding():
    one = 1.0
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa (1.0) wins
    assert orc.round_to_bf16(one + 2.0 ** -8) == 1.0
    # 1 + 3 * 2^-8 is a tie between 1 + 2^-7 (odd) and 1 + 2^-6 (even)
    assert orc.round_to_bf16(one + 3 * 2.0 ** -8) == one + 2.0 ** -6
    # just above the tie in fp64 (an f32 rounding first would land on the tie)
    assert orc.round_to_bf16(one + 2.0 ** -8 + 2.0 ** -40) == one + 2.0 ** -7
    assert orc.round_to_bf16(-(one + 2.0 ** -8 + 2.0 ** -40)) == -(one + 2.0 ** -7)
    assert np.isinf(orc.round_to_bf16(3.4e38))
    assert np.isnan(orc.round_to_bf16(np.nan))


def test_f16_rounding_matches_torch():
    rng = np.random.default_rng(2)
    vals = np.concatenate([rng.standard_normal(20000) * 100, rng.standard_normal(2000) * 1e-6,
                           np.array([65504.0, 65519.9, 65520.0, 2.0 ** -24, 2.0 ** -25])])
    want = torch.from_numpy(vals.astype(np.float32)).to(torch.float16).to(torch.float64).numpy()
    got = orc.round_to_f16(vals.astype(np.float32).astype(np.float64))
    np.testing.assert_array_equal(got, want)


def test_activation_storage_matches_torch():
    # storage in both activation dtypes and the bf16 weight decode, against
    # torch's own dtype conversions of f32 inputs
    rng = np.random.default_rng(3)
    vals = np.concatenate([rng.standard_normal(5000) * 3, rng.standard_normal(500) * 1e-5,
                           np.array([0.0, -0.0, 1.0, -2.5, 65504.0])]).astype(np.float32)
    t = torch.from_numpy(vals)
    want_bf16 = t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got_bf16 = orc.f64_to_act(vals.astype(np.float64), "bf16")
    assert got_bf16.dtype == np.uint16
    np.testing.assert_array_equal(got_bf16, want_bf16)
    np.testing.assert_array_equal(orc.act_to_f64(got_bf16, "bf16"),
                                  t.to(torch.bfloat16).to(torch.float64).numpy())
    np.testing.assert_array_equal(orc.dequant_bf16(got_bf16[:5500].reshape(55, 100)),
                                  t[:5500].to(torch.bfloat16).to(torch.float64).numpy().reshape(55, 100))
    got_f16 = orc.f64_to_act(vals.astype(np.float64), "f16")
    assert got_f16.dtype == np.float16
    np.testing.assert_array_equal(got_f16.view(np.uint16),
                                  t.to(torch.float16).view(torch.int16).numpy().view(np.uint16))
    np.testing.assert_array_equal(orc.act_to_f64(got_f16, "f16"), t.to(torch.float16).to(torch.float64).numpy())
    with pytest.raises(ValueError):
        orc.f64_to_act(vals.astype(np.float64), "f32")


def test_e2m1_e4m3_tables_match_published_values():
    for fmt, code, val in _golden_values():
        fn = orc.e2m1_value if fmt == "e2m1" else orc.e4m3_value
        got = float(fn(code))
        if np.isnan(val):
            assert np.isnan(got), (fmt, code)
        else:
            assert got == val and np.signbit(got) == np.signbit(val), (fmt, hex(code), got, val)


def test_e4m3_all_codes_monotone_and_symmetric():
    pos = orc.e4m3_value(np.arange(0x7F))
    assert np.all(np.diff(pos) > 0)
    neg = orc.e4m3_value(np.arange(0x80, 0xFF))
    np.testing.assert_array_equal(neg, -pos)
    # every finite E4M3 value is exactly a bf16 value (so the product with an
    # E2M1 value is exact in bf16 as well)
    allv = orc.e4m3_value(np.arange(256))
    fin = allv[np.isfinite(allv)]
    prod = (fin[:, None] * orc.e2m1_value(np.arange(16))[None, :]).ravel()
    np.testing.assert_array_equal(orc.round_to_bf16(prod), prod)


def test_gptq_dequant_hand_built_words():
    # one expert, K = 256 (two groups of 128), N = 8
    K, N, G = 256, 8, 128
    qweight = np.zeros((K // 8, N), dtype=np.uint32)
    qweight[0, 0] = 0x76543210          # kappa 0..7 of column 0 hold codes 0..7
    qweight[0, 1] = 0xFEDCBA98          # kappa 0..7 of column 1 hold codes 8..15
    qweight[16, 2] = 0x88888888         # kappa 128..135 of column 2: code 8 == zero
    qweight[15, 3] = 0xF0000000         # kappa 127 (nibble 7 of word 15) of column 3 = 15
    qweight[16, 3] = 0x0000000F         # kappa 128 (nibble 0 of word 16) of column 3 = 15
    scales = np.zeros((K // G, N), dtype=np.float16)
    scales[0, :] = 0.5
    scales[1, :] = 0.25
    qzeros = np.full((K // G, N // 8), 0x88888888, dtype=np.uint32)
    W = orc.dequant_gptq(qweight.view(np.int32), scales, qzeros.view(np.int32), G)   # [N, K]
    assert W.shape == (N, K)
    np.testing.assert_array_equal(W[0, :8], (np.arange(8) - 8) * 0.5)
    np.testing.assert_array_equal(W[1, :8], np.arange(8) * 0.5)
    np.testing.assert_array_equal(W[2, 128:136], np.zeros(8))
    assert W[3, 127] == (15 - 8) * 0.5 and W[3, 128] == (15 - 8) * 0.25
    # code 0 elsewhere: (0 - 8) * scale of the row's group
    assert W[5, 0] == -4.0 and W[5, 200] == -2.0
    # zero points are per column: give column 9 of a wider weight zero 3
    qz2 = np.full((2, 2), 0x88888888, dtype=np.uint32)
    qz2[0, 1] = 0x88888838              # nibble 1 of word 1 -> column 9, group 0
    W2 = orc.dequant_gptq(np.zeros((K // 8, 16), np.int32), np.ones((2, 16), np.float16),
                          qz2.view(np.int32), G)
    assert W2[9, 0] == -3.0 and W2[9, 128] == -8.0 and W2[8, 0] == -8.0


def test_gptq_all_zero_point_codes_give_zero_weight():
    K, N, G = 256, 16, 128
    qw = np.full((K // 8, N), 0x88888888, dtype=np.uint32).view(np.int32)
    sc = np.random.default_rng(0).uniform(0.005, 0.02, (K // G, N)).astype(np.float16)
    qz = np.full((K // G, N // 8), 0x88888888, dtype=np.uint32).view(np.int32)
    assert not orc.dequant_gptq(qw, sc, qz, G).any()


def test_nvfp4_dequant_hand_built_bytes():
    N, K = 2, 32
    packed = np.zeros((N, K // 2), dtype=np.uint8)
    packed[0, 0] = 0x21        # kappa 0 <- low nibble code 1 (0.5), kappa 1 <- code 2 (1.0)
    packed[0, 7] = 0xF7        # kappa 14 <- code 7 (6.0), kappa 15 <- code 15 (-6.0)
    packed[0, 8] = 0x0D        # kappa 16 <- code 13 (-3.0)
    packed[1, 15] = 0x50       # kappa 31 <- code 5 (3.0)
    scales = np.zeros((K // 16, N), dtype=np.uint8)
    scales[0, 0] = 0x38        # 1.0 for kappa 0..15 of row 0
    scales[1, 0] = 0x40        # 2.0 for kappa 16..31 of row 0
    scales[1, 1] = 0x30        # 0.5 for kappa 16..31 of row 1
    W = orc.dequant_nvfp4(packed, scales, np.float32(0.25))
    assert (W[0, 0], W[0, 1], W[0, 14], W[0, 15]) == (0.125, 0.25, 1.5, -1.5)
    assert W[0, 16] == -3.0 * 2.0 * 0.25
    assert W[1, 31] == 3.0 * 0.5 * 0.25 and W[1, 30] == 0.0
    # per-row scale2 (gate rows and up rows of a stacked weight)
    W2 = orc.dequant_nvfp4(packed, scales, np.array([1.0, 4.0], np.float32))
    assert W2[0, 1] == 1.0 and W2[1, 31] == 3.0 * 0.5 * 4.0


def test_expert_weight_nvfp4_gate_up_scale2_split():
    E, N, K = 2, 4, 32
    packed = np.full((E, N, K // 2), 0x22, dtype=np.uint8)        # every element 1.0
    scales = np.full((E, K // 16, N), 0x38, dtype=np.uint8)       # every scale 1.0
    s2 = np.array([[1.0, 2.0], [3.0, 4.0]], np.float32)            # [gate/up, E]
    spec = {"format": "nvfp4", "packed": packed, "scales": scales, "scale2": s2}
    W1 = orc.expert_weight(spec, 1)
    np.testing.assert_array_equal(W1[:2], np.full((2, K), 2.0))   # gate rows: scale2[0, 1]
    np.testing.assert_array_equal(W1[2:], np.full((2, K), 4.0))   # up rows: scale2[1, 1]


def test_prepared_f64_weights_are_the_dequantised_values():
    from mixture_experts_grouped_gb300 import synth
    for wfmt, act in (("bf16", "bf16"), ("gptq", "f16"), ("nvfp4", "bf16"), ("fp8", "bf16")):
        cfg = synth.MoeConfig("p", T=4, H=64, I=64, E=3, k=1, bs=4, wfmt=wfmt, act=act, router="normal",
                              group_size=64)
        w = synth.make_weights(cfg)["w_gate_up"]
        pre = orc.prepare_f64(w)
        for e in range(3):
            np.testing.assert_array_equal(orc.expert_weight(pre, e), orc.expert_weight(w, e))


def test_fp8_dequant_hand_built_codes():
    # 0x38 = 1.0, 0xB8 = -1.0, 0x01 = 2^-9 (smallest subnormal), 0x7E = 448 (largest finite),
    # 0x00 / 0x80 = +0 / -0; row scales 2 and 0.5
    codes = np.array([[0x38, 0xB8, 0x00], [0x01, 0x7E, 0x80]], np.uint8)
    w = orc.dequant_fp8(codes, np.array([2.0, 0.5], np.float32))
    np.testing.assert_array_equal(w, [[2.0, -2.0, 0.0], [2.0 ** -10, 224.0, -0.0]])
    assert np.signbit(w[1, 2])


def test_fp8_dequant_matches_torch_float8():
    # torch's float8_e4m3fn is the OCP E4M3 format: every finite code decodes alike
    codes = np.arange(256, dtype=np.uint8).reshape(16, 16)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = orc.dequant_fp8(codes, np.ones(16, np.float32))
    fin = np.isfinite(want)
    np.testing.assert_array_equal(got[fin], want[fin])
    assert np.all(np.isnan(got[~fin]))


def test_expert_weight_fp8_row_scales():
    from mixture_experts_grouped_gb300 import synth
    cfg = synth.MoeConfig("p", T=4, H=64, I=32, E=3, k=1, bs=4, wfmt="fp8", router="normal")
    w = synth.make_weights(cfg)["w_gate_up"]
    for e in range(3):
        W = orc.expert_weight(w, e)
        assert W.shape == (64, 64)
        np.testing.assert_array_equal(W, orc.e4m3_value(w["codes"][e]) * w["scales"][e].astype(np.float64)[:, None])
        rms = np.sqrt(np.mean(W ** 2))
        assert 0.01 < rms < 0.04 and np.all(np.isfinite(W))
