"""Pins of the oracle's top-k softmax routing (no GPU): brute force, closed
forms, a high-precision evaluation and a library softmax."""
from decimal import Decimal, getcontext

import numpy as np
import pytest
from scipy.special import softmax

import oracle as orc


def _brute_ids(row, k):
    return sorted(range(len(row)), key=lambda i: (-float(row[i]), i))[:k]


@pytest.mark.parametrize("E,k", [(1, 1), (5, 2), (8, 2), (32, 8), (33, 4), (64, 6), (128, 8), (256, 8)])
def test_ids_match_brute_force_sort(E, k):
    rng = np.random.default_rng(E * 31 + k)
    T = 40
    logits = rng.standard_normal((T, E)).astype(np.float32)
    # force ties on half of the rows: small integers repeat often
    logits[::2] = rng.integers(-3, 4, size=(T // 2, E)).astype(np.float32)
    ids, w = orc.route_topk_softmax(logits, k, True)
    for t in range(T):
        assert list(ids[t]) == _brute_ids(logits[t], k)
        assert len(set(ids[t])) == k
        assert np.all(np.diff(w[t]) <= 0), "weights must be non-increasing in rank order"


def _decimal_softmax(vals, sel):
    getcontext().prec = 50
    d = [Decimal(float(v)) for v in vals]
    m = max(d)
    ex = [(v - m).exp() for v in d]
    z = sum(ex[i] for i in sel)
    return [ex[i] / z for i in sel]


@pytest.mark.parametrize("renorm", [True, False])
def test_weights_within_few_ulp_of_high_precision_softmax(renorm):
    rng = np.random.default_rng(7 + renorm)
    for E, k in [(8, 2), (64, 6), (128, 8), (256, 8), (40, 40)]:
        logits = (rng.standard_normal((6, E)) * 3).astype(np.float32)
        ids, w = orc.route_topk_softmax(logits, k, renorm)
        for t in range(logits.shape[0]):
            sel = list(ids[t]) if renorm else list(range(E))
            exact = _decimal_softmax(logits[t], sel)
            if not renorm:
                exact = [exact[sel.index(int(i))] for i in ids[t]]
            n_terms = len(sel)
            for j in range(k):
                ulp = np.spacing(np.float32(exact[j]))
                assert abs(float(w[t, j]) - float(exact[j])) <= (n_terms + 3) * float(ulp)


def test_renormalised_weights_match_library_softmax_of_selected():
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((64, 128)).astype(np.float32)
    ids, w = orc.route_topk_softmax(logits, 8, True)
    for t in range(64):
        ref = softmax(logits[t, ids[t]].astype(np.float64))
        np.testing.assert_allclose(w[t], ref, rtol=2e-6, atol=0)
        assert abs(float(np.sum(w[t], dtype=np.float64)) - 1.0) < 8 * 2 ** -23


def test_unnormalised_weights_match_library_full_softmax():
    rng = np.random.default_rng(4)
    logits = rng.standard_normal((32, 64)).astype(np.float32)
    ids, w = orc.route_topk_softmax(logits, 6, False)
    for t in range(32):
        ref = softmax(logits[t].astype(np.float64))[ids[t]]
        np.testing.assert_allclose(w[t], ref, rtol=1e-5, atol=0)


def test_equal_logits_closed_form():
    E, k = 16, 4
    logits = np.full((3, E), 0.75, dtype=np.float32)
    ids, w = orc.route_topk_softmax(logits, k, True)
    assert np.all(ids == np.arange(k))                      # ties -> lowest indices
    assert np.all(w == np.float32(1.0) / np.float32(k))
    ids, w = orc.route_topk_softmax(logits, k, False)
    assert np.all(w == np.float32(1.0) / np.float32(E))


def test_k_equals_E_is_a_sorted_permutation():
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((10, 12)).astype(np.float32)
    ids, w = orc.route_topk_softmax(logits, 12, True)
    for t in range(10):
        assert sorted(ids[t]) == list(range(12))
        assert np.all(np.diff(logits[t, ids[t]]) <= 0)
        np.testing.assert_allclose(w[t], softmax(logits[t].astype(np.float64))[ids[t]], rtol=2e-6)


def test_two_expert_closed_form():
    # with k = 2 and renormalisation, w0 = 1 / (1 + exp(l1 - l0)) (logistic)
    logits = np.array([[2.0, 0.5, -1.0], [0.0, -3.0, -3.5]], np.float32)
    ids, w = orc.route_topk_softmax(logits, 2, True)
    assert ids.tolist() == [[0, 1], [0, 1]]
    for t in range(2):
        d = float(logits[t, 1]) - float(logits[t, 0])
        assert abs(float(w[t, 0]) - 1.0 / (1.0 + np.exp(d))) < 4e-7
        assert abs(float(w[t, 1]) - np.exp(d) / (1.0 + np.exp(d))) < 4e-7


def test_warp_order_sum_specified_order():
    assert orc.warp_order_sum_f32(np.ones(32, np.float32)) == 32.0
    assert orc.warp_order_sum_f32(np.zeros(0, np.float32)) == 0.0
    v = np.random.default_rng(6).random(256).astype(np.float32)
    s = orc.warp_order_sum_f32(v)
    assert abs(float(s) - float(np.sum(v, dtype=np.float64))) < 256 * 2 ** -24 * 256
    # the order is lane-strided: lane l holds v[l] + v[l + 32] + ...; a vector
    # whose only non-zeros sit in one lane sums exactly left to right
    w = np.zeros(128, np.float32)
    w[[3, 35, 67, 99]] = [1e8, 1.0, -1e8, 1.0]
    want = np.float32(np.float32(np.float32(np.float32(1e8) + np.float32(1.0)) - np.float32(1e8)) + np.float32(1.0))
    assert orc.warp_order_sum_f32(w) == want


def test_invalid_k_rejected():
    with pytest.raises(ValueError):
        orc.route_topk_softmax(np.zeros((2, 4), np.float32), 5, True)
    with pytest.raises(ValueError):
        orc.route_topk_softmax(np.zeros((2, 4), np.float32), 0, True)


def test_router_logits_match_exactly_rounded_sums():
    # every product of a bf16 / fp16 value and an f32 weight is exact in fp64;
    # math.fsum gives the exactly rounded sum, which rounds once to f32
    import math
    from mixture_experts_grouped_gb300 import synth
    for act in ("bf16", "f16"):
        cfg = synth.MoeConfig("r", T=7, H=96, I=8, E=5, k=2, bs=4, act=act, router="gemm", router_std=0.3)
        a = synth.make_activations(cfg)
        got = orc.router_logits(a["x"], act, a["w_router"])
        xf = orc.act_to_f64(a["x"], act)
        wf = a["w_router"].astype(np.float64)
        for t in range(cfg.T):
            for e in range(cfg.E):
                want = np.float32(math.fsum(float(xf[t, h]) * float(wf[h, e]) for h in range(cfg.H)))
                assert got[t, e] == want, (act, t, e, got[t, e], want)
        # the workload's own logits are the same router product
        np.testing.assert_array_equal(got, a["logits"])


def test_router_logits_linear_in_the_weight():
    from mixture_experts_grouped_gb300 import synth
    cfg = synth.MoeConfig("r", T=5, H=64, I=8, E=4, k=1, bs=4, router="gemm", router_std=0.2)
    a = synth.make_activations(cfg)
    w = a["w_router"]
    # a one-hot weight column picks one activation feature exactly
    one = np.zeros_like(w)
    one[17, 2] = 1.0
    got = orc.router_logits(a["x"], "bf16", one)
    np.testing.assert_array_equal(got[:, 2], orc.act_to_f64(a["x"], "bf16")[:, 17].astype(np.float32))
    assert not got[:, [0, 1, 3]].any()
