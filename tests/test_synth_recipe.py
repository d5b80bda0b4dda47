"""The NVFP4 input recipe: block-amax quantisation of a Gaussian.

The workloads' NVFP4 weights are bf16 N(0, 0.02) weights quantised with a
per-expert fp32 scale2 = amax / (6 * 448), E4M3 block scales rounded to
nearest (ties to even) and E2M1 codes rounded the same way. These CPU tests
pin the rounding of the input generator to torch's own E4M3 conversion and to
hand-worked E2M1 midpoints, and check the properties the recipe promises.
"""
import numpy as np
import pytest

import oracle as orc
from mixture_experts_grouped_gb300 import synth


def test_e4m3_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.uniform(0, 448, 20000), np.exp(rng.uniform(np.log(2 ** -12), np.log(448), 20000)),
                        synth._E4M3_VALUES,
                        # exact midpoints between neighbouring codes: ties go to the even code
                        0.5 * (synth._E4M3_VALUES[1:] + synth._E4M3_VALUES[:-1])])
    codes = synth._round_to_table(x, synth._E4M3_VALUES)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(codes, want)


def test_e2m1_rounding_hand_values():
    x = np.array([0.0, 0.2, 0.25, 0.3, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 5.9, 6.0, 7.0, 100.0])
    # midpoints go to the even code: 0.25 -> 0, 0.75 -> 1.0, 1.25 -> 1.0,
    # 1.75 -> 2.0, 2.5 -> 2.0, 3.5 -> 4.0, 5.0 -> 4.0; past 6 saturates
    want = np.array([0, 0, 0, 1, 2, 2, 4, 4, 6, 6, 7, 7, 7, 7], np.uint8)
    np.testing.assert_array_equal(synth._round_to_table(x, synth._E2M1_VALUES), want)


def test_amax_recipe_properties():
    cfg = synth.MoeConfig("q", T=16, H=512, I=256, E=3, k=2, bs=16, wfmt="nvfp4")
    w = synth.make_weights(cfg)
    for key, tensor, groups in (("w_gate_up", synth._GU, 2), ("w_down", synth._DOWN, 1)):
        spec = w[key]
        N, K = spec["packed"].shape[1], 2 * spec["packed"].shape[2]
        rows = N // groups
        for e in range(cfg.E):
            bits = synth._normal_act(synth._rng(cfg.seed, tensor, e), (N, K), cfg.weight_std, "bf16")
            orig = orc.bf16_bits_to_f64(bits)
            codes = np.stack([spec["packed"][e] & 15, spec["packed"][e] >> 4], -1).reshape(N, K)
            # every 16-wide block holds a code of magnitude 6 (amax scaling)
            assert np.all((codes & 7).reshape(N, K // 16, 16).max(axis=2) == 7)
            for g in range(groups):
                sl = slice(g * rows, (g + 1) * rows)
                s2 = spec["scale2"][g, e]
                assert np.isclose(s2, np.float32(np.abs(orig[sl]).max() / (6 * 448)))
                # the largest block of the group gets the largest finite scale, 448
                assert spec["scales"][e][:, sl].max() == 0x7E
                deq = orc.dequant_nvfp4(spec["packed"][e][sl], spec["scales"][e][:, sl], s2)
                rel = np.linalg.norm(deq - orig[sl]) / np.linalg.norm(orig[sl])
                assert rel < 0.12, rel            # 4-bit quantisation of a Gaussian: about 9.5%
                assert np.all(np.sign(deq[deq != 0]) == np.sign(orig[sl][deq != 0]))
