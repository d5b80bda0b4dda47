"""Helpers shared by the GPU parity tests: run a layer through the C ABI and
compare its outputs with the oracle under the stated tolerances."""
from __future__ import annotations

import numpy as np

import oracle as orc

# FFN tolerance: relative Frobenius error and per-element bound
REL_FRO = 5e-3
ELEM = 2e-2


def ffn_close(got: np.ndarray, ref: np.ndarray, what: str = "") -> tuple[float, float]:
    """Assert |got - ref|_F / |ref|_F <= 5e-3 and |got - ref| <= 2e-2 * (1 + |ref|)
    elementwise (fp64 values of activation-rounded numbers)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite GPU values"
    denom = np.linalg.norm(ref)
    fro = float(np.linalg.norm(got - ref) / denom) if denom > 0 else float(np.linalg.norm(got))
    worst = float(np.max(np.abs(got - ref) / (1.0 + np.abs(ref)))) if ref.size else 0.0
    assert fro <= REL_FRO, f"{what}: relative Frobenius error {fro:.3e} > {REL_FRO}"
    assert worst <= ELEM, f"{what}: worst element error {worst:.3e} > {ELEM}"
    return fro, worst


def valid_rows(sorted_ids: np.ndarray, total: int, P: int) -> np.ndarray:
    r = np.arange(total)
    return r[sorted_ids[:total] != P]


def gpu_layer(cfg, inp, device, weights=None, lora=None, row_adapter=None):
    """Build a MoeLayer for cfg, upload inputs, run forward once. Returns
    (layer, x_dev, logits_dev)."""
    import torch
    from mixture_experts_grouped_gb300 import layer as L
    if weights is None:
        weights = (L.upload_weight(inp["w_gate_up"], cfg.act, device), L.upload_weight(inp["w_down"], cfg.act, device))
    dl = None
    if lora is not None:
        dl = L.upload_lora(lora, cfg.I, cfg.H, device)
    ra = None if row_adapter is None else torch.from_numpy(row_adapter.astype(np.int32)).to(device)
    lay = L.MoeLayer(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.bs, cfg.act, weights[0], weights[1], device, lora=dl,
                     renormalize=cfg.renormalize, row_adapter=ra)
    x = L.act_tensor(inp["x"], cfg.act, device)
    logits = torch.from_numpy(inp["logits"]).to(device)
    lay.forward(x, logits)
    torch.cuda.synchronize()
    return lay, x, logits


def fetch(lay):
    from mixture_experts_grouped_gb300 import layer as L
    act = lay.act
    d = {
        "ids": lay.topk_ids.cpu().numpy(),
        "w": lay.topk_weights.cpu().numpy(),
        "sorted": lay.sorted_token_ids.cpu().numpy(),
        "expert_ids": lay.expert_ids.cpu().numpy(),
        "offsets": lay.expert_offsets.cpu().numpy(),
        "total": int(lay.total_post_pad.item()),
        "pair_to_row": lay.pair_to_row.cpu().numpy()[:lay.P],
        "err": int(lay.err.item()),
        "h_bits": L.act_numpy(lay.h, act),
        "y_bits": L.act_numpy(lay.y, act),
        "out_bits": L.act_numpy(lay.out, act),
    }
    d["h"] = orc.act_to_f64(d["h_bits"], act)
    d["y"] = orc.act_to_f64(d["y_bits"], act)
    d["out"] = orc.act_to_f64(d["out_bits"], act)
    return d


def check_route_align_exact(g, ref_ids, ref_w, al):
    assert np.array_equal(g["ids"], ref_ids), "topk ids differ"
    assert np.array_equal(g["w"].view(np.uint32), np.asarray(ref_w, np.float32).view(np.uint32)), \
        f"topk weights differ in {int(np.sum(g['w'] != ref_w))} places"
    assert np.array_equal(g["sorted"], al.sorted_token_ids), "sorted_token_ids differ"
    assert np.array_equal(g["expert_ids"][:al.expert_ids.shape[0]], al.expert_ids), "expert_ids differ"
    assert np.array_equal(g["offsets"], al.expert_offsets), "expert_offsets differ"
    assert g["total"] == al.total_tokens_post_pad
    assert np.array_equal(g["pair_to_row"], al.pair_to_row), "pair_to_row differs"
