"""GPU parity of every step through the C ABI against the CPU oracle.

Routing and align are compared bit for bit; the FFN steps (gate/up, down, LoRA
fold, combine) within relative Frobenius error 5e-3 and per-element
2e-2 * (1 + |ref|). Each FFN step is checked in isolation (the oracle step is
fed the GPU's own input to that step) and the whole layer end to end.
"""
import numpy as np
import pytest

import oracle as orc
from mixture_experts_grouped_gb300 import synth
from parity import check_route_align_exact, fetch, ffn_close, gpu_layer, valid_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mixture_experts_grouped_gb300 import build
    build.build()
    return torch.device("cuda:0")


# ---------------------------------------------------------------------------
# a1 routing: bit-exact
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,E,k,renorm,kind", [
    (16, 8, 2, True, "normal"), (4096, 8, 2, True, "normal"), (517, 128, 8, True, "zipf"),
    (16384, 128, 8, True, "zipf"), (2048, 64, 6, True, "normal"), (300, 256, 16, True, "normal"),
    (300, 256, 16, False, "normal"), (200, 33, 5, False, "ties"), (200, 64, 6, True, "ties"),
    (64, 1, 1, True, "normal"), (1, 128, 8, True, "normal"), (100, 12, 12, False, "normal"),
])
def test_route_bit_exact(dev, T, E, k, renorm, kind):
    import torch
    from mixture_experts_grouped_gb300 import moe
    rng = np.random.default_rng(T * 7 + E)
    if kind == "ties":
        logits = rng.integers(-4, 5, size=(T, E)).astype(np.float32)
    else:
        logits = (rng.standard_normal((T, E)) * 2).astype(np.float32)
        if kind == "zipf":
            logits += (-1.1 * np.log(np.arange(E) + 1.0)).astype(np.float32)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    moe.moe_route_topk_softmax(torch.from_numpy(logits).to(dev), ids, w, T, E, k, renorm)
    torch.cuda.synchronize()
    ref_ids, ref_w = orc.route_topk_softmax(logits, k, renorm)
    np.testing.assert_array_equal(ids.cpu().numpy(), ref_ids)
    got_w = w.cpu().numpy()
    assert np.array_equal(got_w.view(np.uint32), ref_w.view(np.uint32)), \
        f"{int(np.sum(got_w != ref_w))} weights differ; max |d| {np.max(np.abs(got_w - ref_w)):.3e}"


# ---------------------------------------------------------------------------
# a2 align: bit-exact
# ---------------------------------------------------------------------------

def _run_align(dev, ids_np, E, bs, max_padded=None):
    import torch
    from mixture_experts_grouped_gb300 import moe
    P = ids_np.shape[0]
    cap = moe.moe_align_capacity(P, E, bs) if max_padded is None else max_padded
    i32 = dict(dtype=torch.int32, device=dev)
    ids = torch.from_numpy(ids_np.astype(np.int32)).to(dev) if P else torch.empty(1, **i32)
    st = torch.full((max(cap, 1),), -7, **i32)
    eids = torch.full((max(cap // bs, 1),), -7, **i32)
    off = torch.full((E + 1,), -7, **i32)
    tot = torch.full((1,), -7, **i32)
    p2r = torch.full((max(P, 1),), -7, **i32)
    err = torch.zeros(1, **i32)
    wsb = moe.moe_align_workspace_size(P, E)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    moe.moe_align_block_size(ids, P, E, bs, cap, st, eids, off, tot, p2r, err, ws, wsb)
    torch.cuda.synchronize()
    return (st.cpu().numpy()[:cap], eids.cpu().numpy()[:cap // bs], off.cpu().numpy(), int(tot.item()),
            p2r.cpu().numpy()[:P], int(err.item()), cap)


@pytest.mark.parametrize("P,E,bs,skew", [
    (0, 8, 16, 0), (1, 8, 16, 0), (32, 8, 16, 0), (8192, 8, 64, 0), (131072, 128, 64, 1.1),
    (12288, 64, 16, 0), (16384, 128, 64, 0), (5000, 256, 1, 0.5), (3333, 1, 64, 0), (65536, 256, 128, 2.0),
    (2049, 7, 3, 0), (100000, 16, 256, 0.0),
])
def test_align_bit_exact(dev, P, E, bs, skew):
    ids = synth.random_ids(P + E + bs, P, E, skew)
    st, eids, off, tot, p2r, err, cap = _run_align(dev, ids, E, bs)
    ref = orc.align_block_size(ids, E, bs, cap)
    assert err == 0
    np.testing.assert_array_equal(st, ref.sorted_token_ids)
    np.testing.assert_array_equal(eids, ref.expert_ids)
    np.testing.assert_array_equal(off, ref.expert_offsets)
    assert tot == ref.total_tokens_post_pad
    np.testing.assert_array_equal(p2r, ref.pair_to_row)


def test_align_drops_and_flags_out_of_range_ids(dev):
    from mixture_experts_grouped_gb300 import moe
    ids = synth.random_ids(5, 3000, 16, 0)
    ids[[7, 100, 2999]] = [16, -1, 1000]
    st, eids, off, tot, p2r, err, cap = _run_align(dev, ids, 16, 16)
    ref = orc.align_block_size(ids, 16, 16, cap)
    assert err & moe.MOE_DEV_ERR_EXPERT_ID and ref.err == 1
    np.testing.assert_array_equal(st, ref.sorted_token_ids)
    np.testing.assert_array_equal(p2r, ref.pair_to_row)
    np.testing.assert_array_equal(off, ref.expert_offsets)


# ---------------------------------------------------------------------------
# whole layers, each FFN step isolated
# ---------------------------------------------------------------------------

def _cfg(name, **kw):
    base = synth.CONFIGS[name.split("@")[0]]
    if "@" in name:
        base = base.with_T(int(name.split("@T")[1]))
    from dataclasses import replace
    return replace(base, **kw) if kw else base


LAYER_CASES = {
    "tiny": _cfg("tiny"),
    "fine_grained@T1": _cfg("fine_grained@T1"),
    "fine_grained@T8": _cfg("fine_grained@T8"),
    "fine_grained@T64": _cfg("fine_grained@T64"),
    "fine_grained@T512": _cfg("fine_grained@T512"),
    "fine_grained@T1024": _cfg("fine_grained@T1024"),
    "gptq@T16": _cfg("gptq@T16"),
    "gptq@T2048": _cfg("gptq@T2048"),
    # NVFP4 weights from block-amax quantisation of a Gaussian (every 16-wide
    # block holds a code near +-6), decode and prefill forms
    "nvfp4@T64": _cfg("nvfp4_lora@T64", lora_rank=0),
    "nvfp4_lora@T2048": _cfg("nvfp4_lora"),
    # NVFP4 codes and block scales drawn directly (every code, many scale values)
    "nvfp4_drawn@T64": _cfg("nvfp4_lora@T64", lora_rank=0, nvfp4_recipe="draw"),
    "nvfp4_drawn_prefill": synth.MoeConfig("nvfp4_drawn_prefill", T=600, H=256, I=192, E=2, k=1, bs=64,
                                           wfmt="nvfp4", router="normal", nvfp4_recipe="draw"),
    # edge shapes: one expert, ragged I (not a multiple of 128) and a span of several row tiles
    "one_expert_ragged": synth.MoeConfig("one_expert_ragged", T=300, H=128, I=136, E=1, k=1, bs=16,
                                         router="normal"),
    # H below one 256-column output tile, top_k == E, block_size 1
    "small_H_k_eq_E": synth.MoeConfig("small_H_k_eq_E", T=77, H=192, I=64, E=4, k=4, bs=1, router="normal"),
    # skewed: most pairs on one expert (long spans crossing many 128-row tiles)
    "skewed": synth.MoeConfig("skewed", T=1500, H=256, I=256, E=16, k=2, bs=64, router="zipf"),
    "gptq_bf16_act": synth.MoeConfig("gptq_bf16_act", T=40, H=256, I=128, E=8, k=2, bs=16, act="bf16",
                                     wfmt="gptq", router="normal", group_size=64),
    "nvfp4_f16_act": synth.MoeConfig("nvfp4_f16_act", T=40, H=256, I=192, E=8, k=2, bs=16, act="f16",
                                     wfmt="nvfp4", router="normal"),
    # a block size that does not divide the tile height: tiles may start on padding rows
    # (decode form with 64-token tiles, CTA-pair prefill forms for bf16 and GPTQ)
    "block48_decode": synth.MoeConfig("block48_decode", T=200, H=256, I=128, E=8, k=2, bs=48, router="normal"),
    "block48_prefill": synth.MoeConfig("block48_prefill", T=500, H=256, I=256, E=4, k=2, bs=48, router="normal"),
    "block48_gptq": synth.MoeConfig("block48_gptq", T=300, H=256, I=256, E=4, k=2, bs=48, act="f16",
                                    wfmt="gptq", router="normal"),
    # quantised prefill (CTA-pair form) with the other activation type, an odd
    # number of 64-deep k blocks (I=192) and a ragged last column tile (H=320)
    "gptq_bf16_prefill": synth.MoeConfig("gptq_bf16_prefill", T=300, H=320, I=192, E=2, k=1, bs=16, act="bf16",
                                         wfmt="gptq", router="normal", group_size=64),
    "nvfp4_f16_prefill": synth.MoeConfig("nvfp4_f16_prefill", T=300, H=320, I=192, E=2, k=1, bs=16, act="f16",
                                         wfmt="nvfp4", router="normal"),
    # decode form with fewer tiles than SMs: tiles cut into k pieces summed by
    # their owner CTA, with ragged contractions (H=1000, I=520: last k blocks of
    # 40 and 8) and ragged last column tiles
    "splitk_ragged_k": synth.MoeConfig("splitk_ragged_k", T=6, H=1000, I=520, E=4, k=2, bs=16, router="normal"),
    # FP8 (E4M3) weights with row scales: decode (16-token tiles, four issuers), prefill
    # (CTA-pair form) with the other activation type, and a ragged I / K
    "fp8@T64": _cfg("fp8@T64"),
    "fp8_f16_prefill": synth.MoeConfig("fp8_f16_prefill", T=300, H=320, I=208, E=2, k=1, bs=16, act="f16",
                                       wfmt="fp8", router="normal"),
    "fp8_decode_ragged": synth.MoeConfig("fp8_decode_ragged", T=24, H=272, I=144, E=8, k=2, bs=16,
                                         wfmt="fp8", router="normal"),
    # FP8 prefill (the CTA-pair form, 192-row geometry) with bf16 activations, the
    # path of the fp8 workload: >= 128 rows per expert, an odd number of 64-deep k blocks
    # for gate/up (H=320), a ragged last k block for down (I=208) and a
    # ragged last column tile
    "fp8_bf16_prefill": synth.MoeConfig("fp8_bf16_prefill", T=300, H=320, I=208, E=2, k=1, bs=16,
                                        wfmt="fp8", router="normal"),
    # the same at about 300 rows per expert: the CTA-pair form's 256-row geometry
    # (one accumulator buffer, eight weight stages), each expert cut into two row tiles
    "fp8_wide_prefill": synth.MoeConfig("fp8_wide_prefill", T=600, H=320, I=208, E=2, k=1, bs=16,
                                        wfmt="fp8", router="normal"),
    # FP8 decode form with fp16 activations
    "fp8_f16_decode": synth.MoeConfig("fp8_f16_decode", T=24, H=272, I=144, E=8, k=2, bs=16, act="f16",
                                      wfmt="fp8", router="normal"),
    # the fp8 workload at full size (T=2048, E=128, top_k=8: prefill form)
    "fp8@T2048": _cfg("fp8"),
    # CTA-pair form: experts of ~300 rows cut into two tiles of nearly equal height;
    # I=192 leaves the second gate/up column tile half empty
    "pair_tails": synth.MoeConfig("pair_tails", T=600, H=256, I=192, E=2, k=1, bs=16, router="normal"),
    # CTA-pair form with a block size that is not a multiple of 16: a tile's last
    # 16-row unit may run into padding or the next expert's rows, which are not stored
    "pair_bs24": synth.MoeConfig("pair_bs24", T=900, H=320, I=200, E=3, k=2, bs=24, router="normal"),
}


@pytest.mark.parametrize("name", list(LAYER_CASES))
def test_layer_steps_match_oracle(dev, name):
    import torch
    cfg = LAYER_CASES[name]
    inp = synth.make_inputs(cfg)
    lora = inp["lora"]
    lay, x, logits = gpu_layer(cfg, inp, dev, lora=None)   # base path (no fold) first
    g = fetch(lay)
    ref_ids, ref_w = orc.route_topk_softmax(inp["logits"], cfg.k, cfg.renormalize)
    al = orc.align_block_size(ref_ids.reshape(-1), cfg.E, cfg.bs, lay.max_padded)
    check_route_align_exact(g, ref_ids, ref_w, al)
    assert g["err"] == 0, f"device error word {g['err']:#x}"
    # the split-K flags (the last 4 KB of each GEMM workspace) are left zero
    assert not lay.gate_up_ws[-4096:].any() and not lay.down_ws[-4096:].any()
    P = cfg.P
    rows = valid_rows(al.sorted_token_ids, al.total_tokens_post_pad, P)
    # gate/up (+ silu*up) from the same x
    h_ref = orc.grouped_gate_up(inp["x"], cfg.act, inp["w_gate_up"], al.sorted_token_ids, al.expert_offsets, P,
                                cfg.k, cfg.I)
    ffn_close(g["h"][rows], h_ref[rows], f"{name}: h")
    # down from the GPU's own h
    y_ref = orc.grouped_down(g["h"], cfg.act, inp["w_down"], al.sorted_token_ids, al.expert_offsets, P, cfg.H)
    ffn_close(g["y"][rows], y_ref[rows], f"{name}: y")
    # combine from the GPU's own y
    out_ref = orc.combine(g["y"], cfg.act, al.pair_to_row, ref_w, cfg.T, cfg.k)
    ffn_close(g["out"], out_ref, f"{name}: combine")
    if lora is not None:
        # fold in place on the GPU's y, compare with the oracle fold of the same inputs
        from mixture_experts_grouped_gb300 import layer as L
        dl = L.upload_lora(lora, cfg.I, cfg.H, dev)
        lay.lora = dl
        lay.xa = torch.zeros((lay.max_padded, dl.route.max_rank), dtype=torch.bfloat16, device=dev)
        lay.lora_fold()
        torch.cuda.synchronize()
        y_fold = orc.act_to_f64(L.act_numpy(lay.y, cfg.act), cfg.act)
        ref_fold, _ = orc.lora_grouped_down(g["h_bits"], g["y_bits"], lora["a"], lora["b"], lora["scale"],
                                            lora["n_experts"], al.expert_offsets, al.sorted_token_ids, P, cfg.k,
                                            None, 0, al.total_tokens_post_pad)
        ffn_close(y_fold[rows], orc.bf16_bits_to_f64(ref_fold)[rows], f"{name}: LoRA fold")
        # rows of unadapted (odd) experts are untouched, bit for bit
        ex = np.searchsorted(al.expert_offsets, rows, side="right") - 1
        odd = rows[ex % 2 == 1]
        assert np.array_equal(L.act_numpy(lay.y, cfg.act)[odd], g["y_bits"][odd])


@pytest.mark.parametrize("name", ["fine_grained@T1", "fine_grained@T64", "splitk_ragged_k"])
def test_split_k_repeatable(dev, name):
    """Decode launches that cut tiles across CTAs: each run leaves the split-K
    flags zero, so back-to-back runs give the same bits (the owner adds the
    partial sums in a fixed order)."""
    import torch
    cfg = LAYER_CASES[name]
    inp = synth.make_inputs(cfg)
    lay, x, logits = gpu_layer(cfg, inp, dev)
    first = [t.clone() for t in (lay.h, lay.y, lay.out)]
    for _ in range(3):
        lay.forward(x, logits)
    torch.cuda.synchronize()
    assert int(lay.err.item()) == 0
    for a, b in zip(first, (lay.h, lay.y, lay.out)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert not lay.gate_up_ws[-4096:].any() and not lay.down_ws[-4096:].any()


@pytest.mark.parametrize("name", ["fine_grained@T1", "splitk_ragged_k"])
def test_split_k_ignores_stale_areas(dev, name):
    """Split-K partial sums and flags left in the workspaces by an earlier call
    (here: every byte of both split-K areas overwritten with 0x7f, so every
    flag and partial sum is stale) are not taken for the current call's: a
    piece's flags hold the call's generation and the owner accepts only that.
    The outputs are bit-identical to a clean run."""
    import torch
    cfg = LAYER_CASES[name]
    inp = synth.make_inputs(cfg)
    lay, x, logits = gpu_layer(cfg, inp, dev)
    clean = [t.clone() for t in (lay.h, lay.y, lay.out)]
    n = lay.down_ws.numel()  # the down workspace is exactly one split-K area; gate/up's ends with one
    for ws in (lay.gate_up_ws, lay.down_ws):
        ws[-n:].fill_(0x7f)
    lay.forward(x, logits)
    torch.cuda.synchronize()
    assert int(lay.err.item()) == 0
    for what, a, b in zip(("h", "y", "out"), clean, (lay.h, lay.y, lay.out)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"{what} differs from the clean run"


@pytest.mark.parametrize("name", ["tiny", "fine_grained@T64", "gptq@T16", "nvfp4_lora@T2048", "skewed",
                                  "fp8@T2048"])
def test_layer_end_to_end(dev, name):
    cfg = LAYER_CASES[name]
    inp = synth.make_inputs(cfg)
    lay, _, _ = gpu_layer(cfg, inp, dev, lora=inp["lora"])
    g = fetch(lay)
    ref = orc.moe_layer(inp["x"], cfg.act, inp["logits"], cfg.k, cfg.E, cfg.bs, inp["w_gate_up"], inp["w_down"],
                        cfg.I, cfg.H, cfg.renormalize, lora=inp["lora"], max_padded=lay.max_padded)
    check_route_align_exact(g, ref.ids, ref.weights, ref.align)
    ffn_close(g["out"], ref.out, f"{name}: layer output")


@pytest.mark.parametrize("T,H,E,k,act", [(16, 128, 8, 2, "bf16"), (64, 4096, 8, 2, "bf16"), (100, 2048, 128, 8, "bf16"),
                                         (45, 200, 60, 6, "f16"), (33, 1024, 256, 8, "f16"),
                                         (4096, 4096, 8, 2, "bf16"), (300, 2048, 128, 8, "bf16"),
                                         (77, 136, 17, 3, "bf16"), (5, 64, 3, 1, "f16"), (1, 8, 1, 1, "bf16")])
def test_router_gemm_then_routing(dev, T, H, E, k, act):
    """Router GEMM on the GPU: logits within the f32 accumulation bound of the
    oracle's exactly rounded product, and the routing of those logits
    bit-exact (selection, order and weights)."""
    import torch
    from mixture_experts_grouped_gb300 import layer as L, moe
    cfg = synth.MoeConfig("router", T=T, H=H, I=8, E=E, k=k, bs=16, act=act, router="gemm", router_std=0.05)
    a = synth.make_activations(cfg)
    want = orc.router_logits(a["x"], act, a["w_router"]).astype(np.float64)
    xd = L.act_tensor(a["x"], act, dev)
    wd = torch.from_numpy(a["w_router"]).to(dev)
    logits = torch.empty((T, E), dtype=torch.float32, device=dev)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    moe.moe_router_topk_softmax(xd, moe.ACT_CODES[act], wd, T, H, E, k, True, logits, ids, w)
    torch.cuda.synchronize()
    got = logits.cpu().numpy()
    mag = np.abs(orc.act_to_f64(a["x"], act)) @ np.abs(a["w_router"].astype(np.float64))
    assert np.all(np.abs(got - want) <= 2.0 * H * 2.0 ** -24 * mag + 1e-30), float(np.max(np.abs(got - want) / mag))
    ref_ids, ref_w = orc.route_topk_softmax(got, k, True)
    np.testing.assert_array_equal(ids.cpu().numpy(), ref_ids)
    np.testing.assert_array_equal(w.cpu().numpy().view(np.uint32), np.asarray(ref_w, np.float32).view(np.uint32))


@pytest.mark.parametrize("x_gather,adapter,rank,T", [(0, False, 16, 37), (1, True, 16, 37), (0, True, 40, 37),
                                                    (1, False, 64, 37), (0, True, 16, 600), (1, False, 16, 4200)])
def test_lora_gather_bgmv_matches_oracle(dev, x_gather, adapter, rank, T):
    """Decode gather fold on slot-major rows: folded rows within tolerance of the
    oracle, every other row of base and xa untouched bit for bit. Expert ids
    come from real routing; the last adapted expert lies past n_experts. T=600
    (2400 rows) takes the expert-grouped kernel over two compaction segments;
    the others (fewer than 2048 rows, or 16800) the row-per-block kernel."""
    import torch
    from mixture_experts_grouped_gb300 import layer as L, moe
    cfg = synth.MoeConfig("gather_fold", T=T, H=520, I=264, E=16, k=4, bs=16, router="normal",
                          lora_rank=rank, lora_scale=2.0, seed=3)
    inp = synth.make_inputs(cfg)
    lora = dict(inp["lora"])
    lora["n_experts"] = 14                                  # adapted expert 14 folds nothing
    ids, _ = orc.route_topk_softmax(inp["logits"], cfg.k, cfg.renormalize)
    indices = ids.reshape(-1).astype(np.uint32)
    rng = np.random.default_rng(11)
    n = cfg.P
    x = orc.f64_to_bf16_bits(rng.standard_normal((n if x_gather == 0 else cfg.T, cfg.I)))
    base = orc.f64_to_bf16_bits(rng.standard_normal((n, cfg.H)))
    ra = np.where(rng.random(cfg.T) < 0.3, -1, 0).astype(np.int32) if adapter else None
    want, xa_want = orc.lora_gather_bgmv(x, base, lora["a"], lora["b"], lora["scale"], lora["n_experts"],
                                         indices, cfg.k, ra, x_gather)
    dl = L.upload_lora(lora, cfg.I, cfg.H, dev)
    dl.route.n_experts = lora["n_experts"]                   # the table stops before adapted expert 14
    xd = L.act_tensor(x, "bf16", dev)
    bd = L.act_tensor(base, "bf16", dev)
    idx = torch.from_numpy(indices.view(np.int32)).to(dev)
    rad = torch.from_numpy(ra).to(dev) if adapter else None
    xad = torch.zeros((n, dl.route.max_rank), dtype=torch.bfloat16, device=dev)
    moe.moe_lora_gather_bgmv(dl.route, xd, bd, idx, rad, xad, n, cfg.k, x_gather)
    torch.cuda.synchronize()
    got = L.act_numpy(bd, "bf16")
    xa = L.act_numpy(xad, "bf16")
    folded = np.any(want != base, axis=1) | np.any(xa_want != 0, axis=1)
    assert folded.sum() > n // 4 and (~folded).sum() > 0
    np.testing.assert_array_equal(got[~folded], base[~folded])
    assert not xa[~folded].any()
    ffn_close(orc.bf16_bits_to_f64(got[folded]), orc.bf16_bits_to_f64(want[folded]), "gather fold: base")
    ffn_close(orc.bf16_bits_to_f64(xa[folded]), orc.bf16_bits_to_f64(xa_want[folded]), "gather fold: xa")


def test_lora_windows_bit_identical_to_one_window(dev):
    import torch
    from mixture_experts_grouped_gb300 import layer as L
    from mixture_experts_grouped_gb300 import moe
    cfg = _cfg("nvfp4_lora@T256")
    inp = synth.make_inputs(cfg)
    lay, _, _ = gpu_layer(cfg, inp, dev, lora=None)
    dl = L.upload_lora(inp["lora"], cfg.I, cfg.H, dev)
    y0 = lay.y.clone()
    total = int(lay.total_post_pad.item())
    lay.lora, lay.xa = dl, torch.zeros((lay.max_padded, 16), dtype=torch.bfloat16, device=dev)
    lay.lora_fold(row_offset=0, row_end=total)
    one = lay.y.clone()
    for cap in (1, 100, 1000):
        lay.y.copy_(y0)
        xa_small = torch.zeros((cap, 16), dtype=torch.bfloat16, device=dev)
        lay.xa = xa_small
        for lo, hi in moe.lora_windows(total, cap):
            lay.lora_fold(row_offset=lo, row_end=hi)
        torch.cuda.synchronize()
        assert torch.equal(lay.y.view(torch.int16), one.view(torch.int16)), f"cap={cap}"


def test_lora_row_adapter_and_gate_up_gather(dev):
    """row_adapter < 0 skips a token's rows; x_gather = 1 reads token-major rows."""
    import torch
    from mixture_experts_grouped_gb300 import layer as L
    from mixture_experts_grouped_gb300 import moe
    cfg = synth.MoeConfig("lora_gather", T=50, H=128, I=128, E=8, k=2, bs=16, router="normal", lora_rank=8)
    inp = synth.make_inputs(cfg)
    lay, x, _ = gpu_layer(cfg, inp, dev, lora=None)
    g = fetch(lay)
    ra = np.zeros(cfg.T, np.int32)
    ra[::4] = -1
    dl = L.upload_lora(inp["lora"], cfg.I, cfg.H, dev)
    xa = torch.zeros((lay.max_padded, 8), dtype=torch.bfloat16, device=dev)
    ra_d = torch.from_numpy(ra).to(dev)
    for x_gather, src, src_bits in ((0, lay.h, g["h_bits"]), (1, x, inp["x"])):
        base = lay.y.clone()
        moe.moe_lora_grouped_down(dl.route, src, base, lay.expert_offsets, lay.sorted_token_ids, ra_d, xa, 0,
                                  lay.max_padded, x_gather, cfg.T, cfg.k)
        torch.cuda.synchronize()
        al = orc.align_block_size(g["ids"].reshape(-1), cfg.E, cfg.bs, lay.max_padded)
        ref, _ = orc.lora_grouped_down(src_bits, g["y_bits"], inp["lora"]["a"], inp["lora"]["b"],
                                       inp["lora"]["scale"], inp["lora"]["n_experts"], al.expert_offsets,
                                       al.sorted_token_ids, cfg.P, cfg.k, ra, 0, lay.max_padded, x_gather)
        rows = valid_rows(al.sorted_token_ids, al.total_tokens_post_pad, cfg.P)
        got = L.act_numpy(base, "bf16")
        ffn_close(orc.bf16_bits_to_f64(got)[rows], orc.bf16_bits_to_f64(ref)[rows], f"x_gather={x_gather}")
        skipped = rows[ra[al.sorted_token_ids[rows] // cfg.k] < 0]
        assert np.array_equal(got[skipped], g["y_bits"][skipped])


@pytest.mark.parametrize("name", ["tiny", "skewed"])   # decode form, CTA-pair prefill form
def test_gemm_rejects_bad_offsets_on_device(dev, name):
    """expert_offsets that decrease: the GEMM runs no tile and flags the error."""
    import torch
    from mixture_experts_grouped_gb300 import moe
    cfg = LAYER_CASES[name]
    inp = synth.make_inputs(cfg)
    lay, _, _ = gpu_layer(cfg, inp, dev)
    bad = torch.tensor([0, 64, 32] + [96] * (cfg.E - 2), dtype=torch.int32, device=dev)
    lay.err.zero_()
    y_before = lay.y.clone()
    moe.moe_grouped_down(lay.h, lay.act_code, lay.w_down.desc, lay.sorted_token_ids, bad, cfg.T, cfg.k, cfg.H, cfg.I,
                         cfg.E, cfg.bs, lay.max_padded, lay.y, lay.err, lay.down_ws, lay.down_ws_bytes)
    torch.cuda.synchronize()
    assert int(lay.err.item()) & moe.MOE_DEV_ERR_OFFSETS
    assert torch.equal(lay.y.view(torch.int16), y_before.view(torch.int16))


# ---------------------------------------------------------------------------
# full-size workloads: routing/align in full, FFN on sampled tokens
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name,n_sample", [("mixtral_prefill", 24), ("fine_grained@T4096", 48),
                                           ("fine_grained@T16384", 48)])
def test_full_size_sampled(dev, name, n_sample):
    cfg = _cfg(name)
    inp = synth.make_inputs(cfg)
    lay, _, _ = gpu_layer(cfg, inp, dev)
    g = fetch(lay)
    ref_ids, ref_w = orc.route_topk_softmax(inp["logits"], cfg.k, cfg.renormalize)
    al = orc.align_block_size(ref_ids.reshape(-1), cfg.E, cfg.bs, lay.max_padded)
    check_route_align_exact(g, ref_ids, ref_w, al)
    assert g["err"] == 0
    rng = np.random.default_rng(11)
    tokens = np.sort(rng.choice(cfg.T, size=n_sample, replace=False))
    ref = orc.moe_layer(inp["x"], cfg.act, inp["logits"], cfg.k, cfg.E, cfg.bs, inp["w_gate_up"], inp["w_down"],
                        cfg.I, cfg.H, cfg.renormalize, tokens=tokens, max_padded=lay.max_padded)
    pairs = (tokens[:, None] * cfg.k + np.arange(cfg.k)).reshape(-1)
    rows = al.pair_to_row[pairs]
    ffn_close(g["h"][rows], ref.h[rows], f"{name}: sampled h")
    ffn_close(g["y"][rows], ref.y[rows], f"{name}: sampled y")
    ffn_close(g["out"][tokens], ref.out, f"{name}: sampled output")
