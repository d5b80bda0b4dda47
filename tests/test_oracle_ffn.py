"""Pins of the oracle's expert FFN, combine and whole layer (no GPU): a
per-token brute force with exactly rounded sums, dense special cases checked
with torch, and planted mistakes that the brute force must catch."""
import math

import numpy as np
import pytest
import torch

import oracle as orc
from mixture_experts_grouped_gb300 import synth


def _tiny_cfg(**kw):
    base = dict(name="t", T=5, H=16, I=8, E=4, k=2, bs=4, router="normal")
    base.update(kw)
    return synth.MoeConfig(**base)


def brute_force_layer(inp, cfg):
    """Per token, per selected expert: dot products with math.fsum (exactly
    rounded), rounding at the same storage points as the layer, no sorting."""
    act = cfg.act
    x = orc.act_to_f64(inp["x"], act)
    ids, w = orc.route_topk_softmax(inp["logits"], cfg.k, cfg.renormalize)
    Wgu = [orc.expert_weight(inp["w_gate_up"], e) for e in range(cfg.E)]
    Wd = [orc.expert_weight(inp["w_down"], e) for e in range(cfg.E)]
    out = np.zeros((cfg.T, cfg.H))
    for t in range(cfg.T):
        ys = []
        for j in range(cfg.k):
            e = int(ids[t, j])
            h = []
            for n in range(cfg.I):
                g = math.fsum(x[t, c] * Wgu[e][n, c] for c in range(cfg.H))
                u = math.fsum(x[t, c] * Wgu[e][cfg.I + n, c] for c in range(cfg.H))
                h.append(float(orc.round_act(g / (1.0 + math.exp(-g)) * u, act)))
            y = [float(orc.round_act(math.fsum(h[n] * Wd[e][m, n] for n in range(cfg.I)), act))
                 for m in range(cfg.H)]
            ys.append(y)
        for m in range(cfg.H):
            out[t, m] = float(orc.round_act(math.fsum(float(w[t, j]) * ys[j][m] for j in range(cfg.k)), act))
    return out


def _close_to_brute(got, want, act):
    # both sides round the same fp64 quantities; only a value sitting on a
    # rounding boundary may differ, by one unit in the last place
    rel = 2.0 ** -7 if act == "bf16" else 2.0 ** -10
    return np.all(np.abs(got - want) <= rel * np.abs(want) + 1e-30)


@pytest.mark.parametrize("wfmt,act", [("bf16", "bf16"), ("gptq", "f16"), ("nvfp4", "bf16")])
def test_layer_matches_per_token_brute_force(wfmt, act):
    kw = dict(wfmt=wfmt, act=act)
    if wfmt == "gptq":
        kw.update(H=32, I=16, group_size=16)
    if wfmt == "nvfp4":
        kw.update(H=32, I=32)
    cfg = _tiny_cfg(**kw)
    inp = synth.make_inputs(cfg)
    res = orc.moe_layer(inp["x"], act, inp["logits"], cfg.k, cfg.E, cfg.bs, inp["w_gate_up"],
                        inp["w_down"], cfg.I, cfg.H)
    want = brute_force_layer(inp, cfg)
    assert _close_to_brute(res.out, want, act)
    assert np.abs(want).max() > 0


def test_token_subset_matches_full_layer():
    cfg = _tiny_cfg(T=12)
    inp = synth.make_inputs(cfg)
    args = (inp["x"], "bf16", inp["logits"], cfg.k, cfg.E, cfg.bs, inp["w_gate_up"], inp["w_down"], cfg.I, cfg.H)
    full = orc.moe_layer(*args)
    toks = np.array([11, 0, 5])
    part = orc.moe_layer(*args, tokens=toks)
    np.testing.assert_array_equal(part.out, full.out[toks])


def test_single_expert_reduces_to_dense_swiglu_mlp():
    cfg = _tiny_cfg(T=9, H=32, I=24, E=1, k=1, bs=8)
    inp = synth.make_inputs(cfg)
    res = orc.moe_layer(inp["x"], "bf16", inp["logits"], 1, 1, 8, inp["w_gate_up"], inp["w_down"], 24, 32)
    x = torch.from_numpy(orc.bf16_bits_to_f64(inp["x"]))
    wgu = torch.from_numpy(orc.bf16_bits_to_f64(inp["w_gate_up"]["w"][0]))
    wd = torch.from_numpy(orc.bf16_bits_to_f64(inp["w_down"]["w"][0]))
    g = x @ wgu[:24].T
    u = x @ wgu[24:].T
    h = torch.from_numpy(orc.round_to_bf16((torch.nn.functional.silu(g) * u).numpy()))
    y = orc.round_to_bf16((h @ wd.T).numpy())
    assert np.all(res.weights == 1.0)
    np.testing.assert_allclose(res.out, y, rtol=2 ** -7, atol=0)


def test_all_experts_selected_is_the_full_softmax_mixture():
    cfg = _tiny_cfg(T=6, H=16, I=8, E=3, k=3, bs=2)
    inp = synth.make_inputs(cfg)
    res = orc.moe_layer(inp["x"], "bf16", inp["logits"], 3, 3, 2, inp["w_gate_up"], inp["w_down"], 8, 16)
    x = torch.from_numpy(orc.bf16_bits_to_f64(inp["x"]))
    p = torch.softmax(torch.from_numpy(inp["logits"].astype(np.float64)), dim=1)
    mix = torch.zeros(6, 16, dtype=torch.float64)
    for e in range(3):
        wgu = torch.from_numpy(orc.bf16_bits_to_f64(inp["w_gate_up"]["w"][e]))
        wd = torch.from_numpy(orc.bf16_bits_to_f64(inp["w_down"]["w"][e]))
        h = torch.nn.functional.silu(x @ wgu[:8].T) * (x @ wgu[8:].T)
        mix += p[:, e:e + 1] * (h @ wd.T)
    np.testing.assert_allclose(res.out, mix.numpy(), rtol=3e-2, atol=3e-4)


def test_gptq_zero_point_codes_give_zero_output():
    cfg = _tiny_cfg(wfmt="gptq", act="f16", H=32, I=16, group_size=16)
    inp = synth.make_inputs(cfg)
    for key in ("w_gate_up", "w_down"):
        inp[key]["qweight"][:] = np.int32(np.uint32(0x88888888).view(np.int32))
    res = orc.moe_layer(inp["x"], "f16", inp["logits"], cfg.k, cfg.E, cfg.bs, inp["w_gate_up"],
                        inp["w_down"], cfg.I, cfg.H)
    assert not res.out.any()


def test_combine_selects_rows_by_pair_map():
    y = np.arange(12, dtype=np.float64).reshape(6, 2)        # rows of expert outputs
    pair_to_row = np.array([4, 1, -1, 5], np.int32)           # T=2, k=2; pair 2 dropped
    w = np.array([[1.0, 0.0], [0.5, 2.0]], np.float32)
    out = orc.combine(y, "bf16", pair_to_row, w, 2, 2)
    np.testing.assert_array_equal(out, [[8.0, 9.0], [20.0, 22.0]])


# ---------------------------------------------------------------------------
# planted mistakes: each must make the brute-force pin fail
# ---------------------------------------------------------------------------

def _mutated(monkeypatch, which):
    real_gate_up = orc.moe_oracle.grouped_gate_up
    real_down = orc.moe_oracle.grouped_down
    real_route = orc.moe_oracle.route_topk_softmax

    if which == "swap_gate_up":
        def f(x, act, w, sorted_ids, off, P, k, inter, rows=None):
            spec = dict(w)
            wt = np.concatenate([w["w"][:, inter:], w["w"][:, :inter]], axis=1)
            spec["w"] = wt
            return real_gate_up(x, act, spec, sorted_ids, off, P, k, inter, rows)
        monkeypatch.setattr(orc.moe_oracle, "grouped_gate_up", f)
    elif which == "token_is_pair_mod_T":
        def f(x, act, w, sorted_ids, off, P, k, inter, rows=None):
            T = P // k
            s = np.where(sorted_ids == P, P, (sorted_ids % T) * k)
            return real_gate_up(x, act, w, s, off, P, k, inter, rows)
        monkeypatch.setattr(orc.moe_oracle, "grouped_gate_up", f)
    elif which == "transposed_down":
        def f(h, act, w, sorted_ids, off, P, hidden, rows=None):
            spec = dict(w)
            spec["w"] = np.ascontiguousarray(np.transpose(w["w"], (0, 2, 1)))
            return real_down(h, act, spec, sorted_ids, off, P, hidden, rows)
        monkeypatch.setattr(orc.moe_oracle, "grouped_down", f)
    elif which == "weights_unnormalised":
        monkeypatch.setattr(orc.moe_oracle, "route_topk_softmax",
                            lambda lg, k, renorm=True: real_route(lg, k, False))


@pytest.mark.parametrize("which", ["swap_gate_up", "token_is_pair_mod_T", "transposed_down",
                                   "weights_unnormalised"])
def test_planted_mistakes_are_caught(monkeypatch, which):
    cfg = _tiny_cfg(H=16, I=16)
    inp = synth.make_inputs(cfg)
    want = brute_force_layer(inp, cfg)
    _mutated(monkeypatch, which)
    res = orc.moe_oracle.moe_layer(inp["x"], "bf16", inp["logits"], cfg.k, cfg.E, cfg.bs,
                                   inp["w_gate_up"], inp["w_down"], cfg.I, cfg.H)
    assert not _close_to_brute(res.out, want, "bf16")
