"""Pins of the oracle's grouped LoRA fold (no GPU): fold identities, the
merged-weight form, window invariance, adapter masks and the x_gather mode."""
import numpy as np
import pytest
import torch

import oracle as orc
from mixture_experts_grouped_gb300 import synth


def _setup(seed=0, T=24, H=32, I=24, E=6, k=2, bs=4, rank=4, scale=2.0):
    cfg = synth.MoeConfig("lora", T=T, H=H, I=I, E=E, k=k, bs=bs, router="normal",
                          lora_rank=rank, lora_scale=scale, seed=seed)
    inp = synth.make_inputs(cfg)
    res = orc.moe_layer(inp["x"], "bf16", inp["logits"], k, E, bs, inp["w_gate_up"], inp["w_down"], I, H)
    al = res.align
    rows = np.nonzero(al.sorted_token_ids != cfg.P)[0]
    h = np.zeros(res.h.shape, np.uint16)
    y = np.zeros(res.y.shape, np.uint16)
    h[rows] = orc.f64_to_bf16_bits(res.h[rows])
    y[rows] = orc.f64_to_bf16_bits(res.y[rows])
    return cfg, inp, res, al, h, y, rows


def _fold(cfg, inp, al, h, y, row_offset=0, row_end=None, lora=None, row_adapter=None, x_gather=0, x=None):
    lora = lora or inp["lora"]
    row_end = al.total_tokens_post_pad if row_end is None else row_end
    return orc.lora_grouped_down(h if x is None else x, y, lora["a"], lora["b"], lora["scale"], lora["n_experts"],
                                 al.expert_offsets, al.sorted_token_ids, cfg.P, cfg.k, row_adapter,
                                 row_offset, row_end, x_gather)


def _expert_of_rows(al, n):
    e = np.full(n, -1)
    off = al.expert_offsets
    for i in range(off.shape[0] - 1):
        e[off[i]:off[i + 1]] = i
    return e


def test_zero_scale_leaves_base_bit_identical():
    cfg, inp, res, al, h, y, rows = _setup()
    lora = dict(inp["lora"])
    lora["scale"] = np.zeros_like(lora["scale"])
    out, _ = _fold(cfg, inp, al, h, y, lora=lora)
    np.testing.assert_array_equal(out, y)


def test_zero_A_leaves_base_bit_identical():
    cfg, inp, res, al, h, y, rows = _setup()
    lora = dict(inp["lora"])
    lora["a"] = {e: np.zeros_like(a) for e, a in lora["a"].items()}
    out, xa = _fold(cfg, inp, al, h, y, lora=lora)
    np.testing.assert_array_equal(out, y)
    assert not xa.any()


def test_unadapted_experts_rows_unchanged_and_adapted_rows_change():
    cfg, inp, res, al, h, y, rows = _setup()
    out, _ = _fold(cfg, inp, al, h, y)
    ex = _expert_of_rows(al, y.shape[0])
    odd = rows[ex[rows] % 2 == 1]
    even = rows[ex[rows] % 2 == 0]
    np.testing.assert_array_equal(out[odd], y[odd])
    assert np.mean(np.any(out[even] != y[even], axis=1)) > 0.9


def test_fold_matches_merged_dense_weight():
    # y_folded ~ h (Wd + s B A)^T: the fold is a rank-r update of the down weight
    cfg, inp, res, al, h, y, rows = _setup(scale=8.0)
    out, _ = _fold(cfg, inp, al, h, y)
    ex = _expert_of_rows(al, y.shape[0])
    hv = torch.from_numpy(orc.bf16_bits_to_f64(h))
    got = orc.bf16_bits_to_f64(out)
    for e in range(cfg.E):
        r = rows[ex[rows] == e]
        if r.size == 0:
            continue
        Wd = torch.from_numpy(orc.expert_weight(inp["w_down"], e))
        if e in inp["lora"]["a"]:
            A = torch.from_numpy(orc.bf16_bits_to_f64(inp["lora"]["a"][e]))
            B = torch.from_numpy(orc.bf16_bits_to_f64(inp["lora"]["b"][e]))
            Wd = Wd + 8.0 * (B @ A)
        want = (hv[r] @ Wd.T).numpy()
        err = np.linalg.norm(got[r] - want) / np.linalg.norm(want)
        assert err < 1e-2, (e, err)


@pytest.mark.parametrize("cap", [1, 3, 7, 16, 1000])
def test_windows_are_bit_identical_to_one_full_window(cap):
    cfg, inp, res, al, h, y, rows = _setup(seed=1)
    full, xa_full = _fold(cfg, inp, al, h, y)
    cur = y.copy()
    total = al.total_tokens_post_pad
    for lo in range(0, total, cap):
        hi = min(lo + cap, total)
        cur, xa = _fold(cfg, inp, al, h, cur, lo, hi)
        assert xa.shape[0] == hi - lo
        # xa is indexed by the local row r - row_offset
        np.testing.assert_array_equal(xa, xa_full[lo:hi])
    np.testing.assert_array_equal(cur, full)


def test_row_adapter_negative_skips_token():
    cfg, inp, res, al, h, y, rows = _setup(seed=2)
    ra = np.zeros(cfg.T, np.int32)
    ra[::3] = -1
    out, _ = _fold(cfg, inp, al, h, y, row_adapter=ra)
    full, _ = _fold(cfg, inp, al, h, y)
    toks = al.sorted_token_ids[rows] // cfg.k
    skip = rows[ra[toks] < 0]
    keep = rows[ra[toks] >= 0]
    np.testing.assert_array_equal(out[skip], y[skip])
    np.testing.assert_array_equal(out[keep], full[keep])


def test_n_experts_bounds_the_table():
    cfg, inp, res, al, h, y, rows = _setup(seed=3)
    lora = dict(inp["lora"])
    lora["n_experts"] = 2          # only expert 0 (adapted) and 1 (not) are looked at
    out, _ = _fold(cfg, inp, al, h, y, lora=lora)
    ex = _expert_of_rows(al, y.shape[0])
    beyond = rows[ex[rows] >= 2]
    np.testing.assert_array_equal(out[beyond], y[beyond])
    e0 = rows[ex[rows] == 0]
    assert np.any(out[e0] != y[e0])


def test_x_gather_reads_token_major_rows():
    # x_gather = 1: the shrink input row is x[token of the pair]; compare with
    # x_gather = 0 on an explicitly gathered copy
    cfg, inp, res, al, h, y, rows = _setup(seed=4, H=32, I=32)
    x_tok = inp["x"]                                   # [T, H] with H == I here
    gathered = np.zeros((y.shape[0], cfg.H), np.uint16)
    gathered[rows] = x_tok[al.sorted_token_ids[rows] // cfg.k]
    lora = dict(inp["lora"])
    a, _ = _fold(cfg, inp, al, h, y, x_gather=1, x=x_tok, lora=lora)
    b, _ = _fold(cfg, inp, al, h, y, x_gather=0, x=gathered, lora=lora)
    np.testing.assert_array_equal(a, b)


def test_fold_step_rounds_in_f32_without_fma():
    # one row, rank 1: base = 1.0, delta = 2^-9 (after rounding), scale = 1.5
    # f32(1.0 + 1.5 * 2^-9) = 1.0029296875 is below half a bf16 step above 1.0
    sorted_ids = np.array([0], np.int32)
    off = np.array([0, 1], np.int32)
    x = orc.f64_to_bf16_bits(np.array([[1.0]]))
    base = orc.f64_to_bf16_bits(np.array([[1.0]]))
    A = {0: orc.f64_to_bf16_bits(np.array([[1.0]]))}
    B = {0: orc.f64_to_bf16_bits(np.array([[2.0 ** -9]]))}
    out, xa = orc.lora_grouped_down(x, base, A, B, np.array([1.5], np.float32), 1, off, sorted_ids, 1, 1,
                                    None, 0, 1)
    assert orc.bf16_bits_to_f64(xa)[0, 0] == 1.0
    assert orc.bf16_bits_to_f64(out)[0, 0] == 1.0
    # scale 3: 1 + 3 * 2^-9 = 1.005859375 -> nearest bf16 is 1 + 2^-7 = 1.0078125
    out, _ = orc.lora_grouped_down(x, base, A, B, np.array([3.0], np.float32), 1, off, sorted_ids, 1, 1,
                                   None, 0, 1)
    assert orc.bf16_bits_to_f64(out)[0, 0] == 1.0078125


# ---------------------------------------------------------------------------
# decode gather fold (slot-major rows)
# ---------------------------------------------------------------------------

def _slot_setup(seed=5):
    cfg, inp, res, al, h, y, rows = _setup(seed=seed)
    rng = np.random.default_rng(seed)
    n_slots = cfg.P
    k_in = cfg.I
    indices = res.ids.reshape(-1).astype(np.uint32)              # expert of slot s = t*k + j
    p2r = al.pair_to_row
    base_slot = orc.f64_to_bf16_bits(rng.standard_normal((n_slots, cfg.H)))
    x_slot = orc.f64_to_bf16_bits(rng.standard_normal((n_slots, k_in)))
    x_tok = orc.f64_to_bf16_bits(rng.standard_normal((cfg.T, k_in)))
    return cfg, inp, al, indices, p2r, base_slot, x_slot, x_tok


def _sorted_copy(al, slot_rows, n_rows):
    out = np.zeros((n_rows,) + slot_rows.shape[1:], slot_rows.dtype)
    out[al.pair_to_row] = slot_rows
    return out


@pytest.mark.parametrize("x_gather", [0, 1])
def test_gather_fold_equals_sorted_fold_on_the_same_pairs(x_gather):
    # the slot-major fold of row s is the sorted fold of the row holding pair s
    cfg, inp, al, indices, p2r, base_slot, x_slot, x_tok = _slot_setup()
    lora = inp["lora"]
    n_rows = al.sorted_token_ids.shape[0]
    base_sorted = _sorted_copy(al, base_slot, n_rows)
    x = x_slot if x_gather == 0 else x_tok
    xs = _sorted_copy(al, x_slot, n_rows) if x_gather == 0 else x_tok
    got, xa = orc.lora_gather_bgmv(x, base_slot, lora["a"], lora["b"], lora["scale"], lora["n_experts"],
                                   indices, cfg.k, None, x_gather)
    want, xa_want = orc.lora_grouped_down(xs, base_sorted, lora["a"], lora["b"], lora["scale"], lora["n_experts"],
                                          al.expert_offsets, al.sorted_token_ids, cfg.P, cfg.k, None, 0,
                                          al.total_tokens_post_pad, x_gather)
    np.testing.assert_array_equal(got, want[p2r])
    np.testing.assert_array_equal(xa, xa_want[p2r])
    # adapted experts (even) changed their rows, the others did not
    even = indices % 2 == 0
    assert np.all(np.any(got[even] != base_slot[even], axis=1))
    np.testing.assert_array_equal(got[~even], base_slot[~even])


def test_gather_fold_row_adapter_is_per_token():
    cfg, inp, al, indices, p2r, base_slot, x_slot, x_tok = _slot_setup(seed=6)
    lora = inp["lora"]
    ra = np.zeros(cfg.T, np.int32)
    ra[1::2] = -1                                              # odd tokens keep their base rows
    got, _ = orc.lora_gather_bgmv(x_slot, base_slot, lora["a"], lora["b"], lora["scale"], lora["n_experts"],
                                  indices, cfg.k, ra, 0)
    full, _ = orc.lora_gather_bgmv(x_slot, base_slot, lora["a"], lora["b"], lora["scale"], lora["n_experts"],
                                   indices, cfg.k, None, 0)
    tok = np.arange(cfg.P) // cfg.k
    np.testing.assert_array_equal(got[tok % 2 == 1], base_slot[tok % 2 == 1])
    np.testing.assert_array_equal(got[tok % 2 == 0], full[tok % 2 == 0])


def test_gather_fold_skips_experts_past_the_table():
    cfg, inp, al, indices, p2r, base_slot, x_slot, x_tok = _slot_setup(seed=7)
    lora = inp["lora"]
    got, xa = orc.lora_gather_bgmv(x_slot, base_slot, lora["a"], lora["b"], lora["scale"], 2,
                                   indices, cfg.k, None, 0)
    keep = indices != 0                                        # only expert 0 is adapted and < 2
    np.testing.assert_array_equal(got[keep], base_slot[keep])
    assert not xa[keep].any()
    assert np.all(np.any(got[~keep] != base_slot[~keep], axis=1))


def test_gather_fold_single_row_by_hand():
    # one slot, rank 1, k_in 2, n_out 2, all values exact in bf16:
    # xa = 1*2 + 3*(-1) = -1; delta = [-1 * 4, -1 * 0.5] = [-4, -0.5];
    # base' = base + 2 * delta = [10 - 8, 1 - 1] = [2, 0]
    b = orc.f64_to_bf16_bits
    got, xa = orc.lora_gather_bgmv(b(np.array([[1.0, 3.0]])), b(np.array([[10.0, 1.0]])),
                                   {0: b(np.array([[2.0, -1.0]]))}, {0: b(np.array([[4.0], [0.5]]))},
                                   np.array([2.0], np.float32), 1, np.array([0], np.uint32), 1, None, 0)
    np.testing.assert_array_equal(orc.bf16_bits_to_f64(got), [[2.0, 0.0]])
    np.testing.assert_array_equal(orc.bf16_bits_to_f64(xa), [[-1.0]])


def test_gather_bgmv_grids_of_the_page():
    # four outputs per block along x, one slot per block along y
    assert orc.gather_bgmv_grids(16, 2048, 64) == ([4, 64, 1], [512, 64, 1])
    assert orc.gather_bgmv_grids(17, 2050, 1) == ([5, 1, 1], [513, 1, 1])
