"""Plain numpy oracle of the grouped MoE expert-FFN path (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this module. It shares no code with the CUDA library or its binding.

Each public function cites the page and item it restates. Page keys:

* [lora]   ``spark_model/layers/ops/moe_lora_grouped.rs``
* [ferrum] ``ferrum-kernels 0.7.7, src/backend/cuda/moe.rs``
* [triton] ``ferrum-kernels, src/backend/cuda/triton_fused_moe.rs``
* [cutlass] ``metrale_gpu_runtime/cutlass/grouped.rs``

Conventions (readings of the pages, listed in the design notes):

* A pair id is ``p = t * top_k + j`` (token t, slot j). ``sorted_token_ids``
  holds pair ids and its sentinel is ``P = T * top_k`` ([triton] module doc:
  "sentinel ``total_pairs`` for padding"). The owning token is ``p // top_k``
  ([lora] ``gather_row_token``).
* ``expert_offsets`` is the padded prefix sum of per-expert spans, each span a
  multiple of ``block_size``; expert e owns sorted rows
  ``[expert_offsets[e], expert_offsets[e+1])`` ([cutlass] ``nvfp4_grouped_down``
  doc, [lora] ``moe_lora_grouped_down`` doc).
* bf16 and fp16 tensors are held as raw ``uint16`` bit patterns / ``float16``.
* Weights are indexed ``W[n, kappa]`` (output feature n, contraction index
  kappa) after dequantisation, whatever their storage layout.
"""

from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Callable, Optional, Sequence, Tuple

import numpy as np

__all__ = [
    "bf16_bits_to_f64", "round_to_bf16", "f64_to_bf16_bits", "round_to_f16",
    "round_act", "act_to_f64", "f64_to_act",
    "align_capacity", "router_logits", "route_topk_softmax", "warp_order_sum_f32",
    "align_block_size", "AlignResult", "ensure_group_arrays", "GroupArrayError",
    "e2m1_value", "e4m3_value", "dequant_bf16", "dequant_gptq", "dequant_nvfp4", "dequant_fp8",
    "expert_weight", "prepare_f64", "grouped_gate_up", "grouped_down", "lora_grouped_down",
    "lora_gather_bgmv", "gather_bgmv_grids", "combine", "moe_layer", "LayerResult",
]

# ----------------------------------------------------------------------------
# Number formats
# ----------------------------------------------------------------------------

_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact fp64 values (bf16 is the top half of f32)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return u.view(np.float32).astype(np.float64)


def round_to_bf16(x) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value, ties to even (one rounding).

    bf16 keeps 8 significant bits and f32's exponent range: a value
    ``m * 2**e`` with ``0.5 <= |m| < 1`` is a multiple of ``2**(e-8)``; below
    the smallest normal (2**-126) the step is fixed at 2**-133. Overflow past
    the largest finite value rounds to infinity.
    """
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(invalid="ignore", over="ignore"):
        _, e = np.frexp(x)
        step = np.ldexp(1.0, np.maximum(e, -125) - 8)
        r = np.rint(x / step) * step
        r = np.where(np.isfinite(x) & (np.abs(r) > _BF16_MAX), np.copysign(np.inf, x), r)
    return r


def f64_to_bf16_bits(x) -> np.ndarray:
    """fp64 -> bf16 bit patterns (uint16), rounding once to nearest-even."""
    r = round_to_bf16(x).astype(np.float32)  # exact: r is a bf16 value
    return (r.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def round_to_f16(x) -> np.ndarray:
    """Round fp64 values to the nearest fp16 value, ties to even (numpy's direct
    double -> half conversion), returned as fp64."""
    with np.errstate(over="ignore"):
        return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def round_act(x, act: str) -> np.ndarray:
    """Round to the activation dtype ('bf16' or 'f16'), returned as fp64 values."""
    if act == "bf16":
        return round_to_bf16(x)
    if act == "f16":
        return round_to_f16(x)
    raise ValueError(f"unknown activation dtype {act!r}")


def act_to_f64(a: np.ndarray, act: str) -> np.ndarray:
    """Activation storage (uint16 bf16 bits or float16) -> fp64 values."""
    if act == "bf16":
        return bf16_bits_to_f64(a)
    if act == "f16":
        return np.asarray(a, dtype=np.float16).astype(np.float64)
    raise ValueError(f"unknown activation dtype {act!r}")


def f64_to_act(x: np.ndarray, act: str) -> np.ndarray:
    """fp64 values -> activation storage (uint16 bf16 bits or float16)."""
    if act == "bf16":
        return f64_to_bf16_bits(x)
    if act == "f16":
        return np.asarray(x, dtype=np.float64).astype(np.float16)
    raise ValueError(f"unknown activation dtype {act!r}")


# ----------------------------------------------------------------------------
# Step a1: top-k softmax routing
# ----------------------------------------------------------------------------

def warp_order_sum_f32(v: np.ndarray) -> np.float32:
    """The f32 sum of ``v`` in one fixed order: 32 lane partials (lane l adds
    v[l], v[l+32], ... left to right from 0.0), then pairwise xor-butterfly
    steps 16, 8, 4, 2, 1. This is the order a one-warp-per-row router reduces
    in ([ferrum] ``route_topk_softmax``: "one warp (32 threads), one block per
    row"); the pages do not print the kernel, so the order is a stated reading.
    """
    v = np.asarray(v, dtype=np.float32)
    part = [np.float32(0.0)] * 32
    for i in range(v.shape[0]):
        part[i % 32] = np.float32(part[i % 32] + v[i])
    for off in (16, 8, 4, 2, 1):
        part = [np.float32(part[l] + part[l ^ off]) for l in range(32)]
    return part[0]


def router_logits(x: np.ndarray, act: str, w_router: np.ndarray) -> np.ndarray:
    """Router GEMM before step a1: ``logits[t, e] = f32(sum_h x[t, h] *
    Wr[h, e])`` with the sum taken in fp64 and rounded once to f32.

    The pages route from given logits and print no router; the workloads
    define one (a router weight ``Wr [H, E]`` f32 and logits computed once on
    the host from the activations). ``x`` holds bf16 bits or fp16 values
    (``act``); every product is exact in fp64.
    """
    xf = act_to_f64(np.asarray(x), act)
    return (xf @ np.asarray(w_router, dtype=np.float32).astype(np.float64)).astype(np.float32)


def route_topk_softmax(logits: np.ndarray, top_k: int, renormalize: bool = True):
    """Top-k softmax routing ([ferrum] ``route_topk_softmax``).

    Per row of f32 logits ``[T, E]``: pick the ``top_k`` experts with the largest
    logits (equal logits: lower expert index first), in descending order, and
    give each the softmax probability; with ``renormalize`` (the page's
    ``norm_topk_prob``) the k probabilities are rescaled to sum to one.

    f32 arithmetic (the page keeps a per-row probability vector in fp32 and the
    weights come back as ``Vec<f32>``):  ``d_i = l_i - max`` in f32;
    ``e_i = f32(exp(d_i))`` with the exponential evaluated in fp64 and rounded
    once; renormalised: ``S = e_id0 + e_id1 + ...`` in f32 in rank order and
    ``w_j = e_idj / S`` (IEEE f32 division); otherwise ``Z`` is the f32 sum of
    all ``e_i`` in :func:`warp_order_sum_f32` order and ``w_j = e_idj / Z``.

    Returns ``ids [T, top_k] int32`` and ``weights [T, top_k] float32``.
    """
    lg = np.asarray(logits, dtype=np.float32)
    T, E = lg.shape
    if not (1 <= top_k <= E):
        raise ValueError(f"top_k={top_k} must be in [1, E={E}]")
    ids = np.empty((T, top_k), dtype=np.int32)
    w = np.empty((T, top_k), dtype=np.float32)
    index = np.arange(E)
    for t in range(T):
        row = lg[t]
        # lexsort: last key is primary -> descending logit, then ascending index
        order = np.lexsort((index, -row))
        top = order[:top_k]
        m = row[order[0]]
        d = (row - m).astype(np.float32)                       # f32 subtraction
        e = np.exp(d.astype(np.float64)).astype(np.float32)    # one rounding to f32
        if renormalize:
            s = np.float32(0.0)
            for j in top:
                s = np.float32(s + e[j])
        else:
            s = warp_order_sum_f32(e)
        ids[t] = top
        w[t] = [np.float32(e[j] / s) for j in top]
    return ids, w


# ----------------------------------------------------------------------------
# Step a2: align pairs into block-padded per-expert spans
# ----------------------------------------------------------------------------

def align_capacity(P: int, E: int, block_size: int) -> int:
    """Worst-case padded row count: ``round_up(P + min(E, P) * (bs - 1), bs)``.

    Every non-empty expert pads its span by at most ``bs - 1`` rows, and at most
    ``min(E, P)`` experts are non-empty. Plays the role of the page's
    ``sorted_max_size`` ([ferrum] ``moe_align_block_size``).
    """
    if block_size <= 0:
        raise ValueError("block_size must be positive")
    raw = P + min(E, P) * (block_size - 1)
    return -(-raw // block_size) * block_size


@dataclass
class AlignResult:
    sorted_token_ids: np.ndarray   # [max_padded] int32, pair ids, sentinel P
    expert_ids: np.ndarray         # [max_padded // bs] int32, -1 past the total
    expert_offsets: np.ndarray     # [E + 1] int32 padded prefix sum
    total_tokens_post_pad: int
    pair_to_row: np.ndarray        # [P] int32, -1 for dropped pairs
    err: int                       # 1 if any id was outside [0, E)


def align_block_size(topk_ids: np.ndarray, num_experts: int, block_size: int,
                     max_padded: Optional[int] = None) -> AlignResult:
    """Sort (token, expert) pairs into per-expert spans padded to ``block_size``.

    Restates [ferrum] ``moe_align_block_size`` / ``moe_align_block_size_pair_ids``
    (outputs ``sorted_token_ids``, ``block_ids`` = ``expert_ids`` one per block,
    ``total_tokens_post_pad``) and ``moe_build_pairs_by_token`` (the pair ->
    row map and the ``expert_offsets`` prefix), with pair ids as the sorted
    entries and ``P`` as the sentinel ([triton] module doc).

    * ``c_e`` = number of pairs routed to e; span ``s_e = ceil(c_e / bs) * bs``
      (an empty expert gets no rows).
    * ``expert_offsets[0] = 0``, ``expert_offsets[e+1] = expert_offsets[e] + s_e``,
      total = ``expert_offsets[E]``.
    * Within a span, pairs keep ascending pair order (a stable sort), then
      sentinel rows ``P`` pad the span; rows ``[total, max_padded)`` hold ``P``.
    * ``expert_ids[b] = e`` for every block b of e's span, ``-1`` past the
      total (the page treats ids < 0 as inactive blocks).
    * Ids outside ``[0, E)`` are dropped and flagged in ``err``.
    """
    ids = np.asarray(topk_ids, dtype=np.int64).reshape(-1)
    P = ids.shape[0]
    E, bs = int(num_experts), int(block_size)
    if max_padded is None:
        max_padded = align_capacity(P, E, bs)
    valid = (ids >= 0) & (ids < E)
    counts = np.bincount(ids[valid], minlength=E) if E > 0 else np.zeros(0, np.int64)
    spans = -(-counts // bs) * bs
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(spans)
    total = int(offsets[E])
    if total > max_padded:
        raise ValueError(f"padded total {total} exceeds max_padded {max_padded}")
    sorted_ids = np.full(max_padded, P, dtype=np.int64)
    expert_ids = np.full(max_padded // bs, -1, dtype=np.int64)
    pair_to_row = np.full(P, -1, dtype=np.int64)
    for e in range(E):
        pairs = np.nonzero(ids == e)[0]          # ascending pair ids: stable
        rows = offsets[e] + np.arange(pairs.shape[0])
        sorted_ids[rows] = pairs
        pair_to_row[pairs] = rows
        expert_ids[offsets[e] // bs: offsets[e + 1] // bs] = e
    return AlignResult(sorted_ids.astype(np.int32), expert_ids.astype(np.int32),
                       offsets.astype(np.int32), total, pair_to_row.astype(np.int32),
                       0 if bool(valid.all()) else 1)


class GroupArrayError(ValueError):
    pass


def ensure_group_arrays(who: str, num_experts: int,
                        per_expert: Sequence[Tuple[str, int]],
                        offsets: Sequence[int]) -> None:
    """The grouped-launch argument rules of [cutlass] ``ensure_group_arrays``:
    ``offsets`` has ``num_experts + 1`` entries, every per-expert array has
    exactly ``num_experts`` entries (the message names the array and its
    length), ``offsets[0] >= 0`` and the offsets never decrease (equal
    neighbours are an empty expert). The upper bound is the caller's check."""
    if len(offsets) != num_experts + 1:
        raise GroupArrayError(
            f"{who}: expert_offsets len {len(offsets)} != num_experts+1 {num_experts + 1}")
    for name, n in per_expert:
        if n != num_experts:
            raise GroupArrayError(f"{who}: {name} len {n} != num_experts {num_experts}")
    if offsets[0] < 0:
        raise GroupArrayError(f"{who}: expert_offsets[0] = {offsets[0]} is negative")
    for a, b in zip(offsets[:-1], offsets[1:]):
        if b < a:
            raise GroupArrayError(f"{who}: expert_offsets is not non-decreasing ({a} then {b})")


# ----------------------------------------------------------------------------
# Weight formats (dequantisation)
# ----------------------------------------------------------------------------

def e2m1_value(code) -> np.ndarray:
    """FP4 E2M1 (OCP microscaling element type): sign bit 3, exponent bits 2..1
    (bias 1), mantissa bit 0; exponent 0 is subnormal (0 or 0.5)."""
    c = np.asarray(code, dtype=np.int64) & 0xF
    s = np.where((c >> 3) & 1, -1.0, 1.0)
    e = (c >> 1) & 3
    m = c & 1
    mag = np.where(e == 0, 0.5 * m, np.ldexp(1.0 + 0.5 * m, e - 1))
    return s * mag


def e4m3_value(code) -> np.ndarray:
    """FP8 E4M3 (OCP 8-bit floating point, 'fn' variant): sign bit 7, exponent
    bits 6..3 (bias 7), mantissa bits 2..0; no infinities, 0x7F/0xFF are NaN;
    exponent 0 is subnormal with step 2**-9."""
    c = np.asarray(code, dtype=np.int64) & 0xFF
    s = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 7
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return s * mag


def dequant_bf16(w_e: np.ndarray) -> np.ndarray:
    """bf16 weight ``[N, K]`` (bit patterns) -> fp64 ``W[n, kappa]``."""
    return bf16_bits_to_f64(w_e)


def dequant_gptq(qweight: np.ndarray, scales: np.ndarray, qzeros: np.ndarray,
                 group_size: int) -> np.ndarray:
    """Raw GPTQ 4-bit weight of one expert -> fp64 ``W[n, kappa]``.

    Layout from [triton] ``TritonStackedGptqWeight`` / ``load_stacked_gptq_raw``
    (bits must be 4): ``qweight [K/8, N]`` int32, ``scales [K/G, N]`` fp16,
    ``qzeros [K/G, N/8]`` int32. Readings (the page does not print the kernel):
    nibble j (bits 4j..4j+3) of ``qweight[i, n]`` holds ``q[8i + j, n]``; nibble
    ``n % 8`` of ``qzeros[g, n // 8]`` holds the zero point of column n in group
    g, used as stored; ``w[kappa, n] = (q - z) * s[kappa // G, n]``.
    """
    qw = np.asarray(qweight).astype(np.int64) & 0xFFFFFFFF
    K8, N = qw.shape
    K = K8 * 8
    shifts = (4 * np.arange(8)).reshape(1, 8, 1)
    q = ((qw[:, None, :] >> shifts) & 0xF).reshape(K, N)            # q[kappa, n]
    qz = np.asarray(qzeros).astype(np.int64) & 0xFFFFFFFF
    G = K // group_size
    z = ((qz[:, :, None] >> shifts.reshape(1, 1, 8)) & 0xF).reshape(G, N)  # z[g, n]
    s = np.asarray(scales, dtype=np.float16).astype(np.float64)            # s[g, n]
    grp = np.arange(K) // group_size
    w_kn = (q - z[grp, :]).astype(np.float64) * s[grp, :]
    return w_kn.T.copy()


def dequant_nvfp4(packed: np.ndarray, scales: np.ndarray, scale2) -> np.ndarray:
    """NVFP4 weight of one expert -> fp64 ``W[n, kappa]``.

    Layout from [cutlass] ``nvfp4_grouped_gate_up`` doc: packed E2M1 ``[N, K/2]``
    and E4M3 block scales ``[K/16, N]`` (one scale per 16 contraction elements),
    plus the per-expert fp32 ``scale2``. Readings: byte ``(n, kappa // 2)``
    holds even kappa in its low nibble, odd kappa in its high nibble;
    ``w = e2m1 * e4m3(scale[kappa // 16, n]) * scale2``. ``scale2`` may be a
    scalar or a per-row ``[N]`` vector (gate and up rows carry their own).
    """
    pk = np.asarray(packed, dtype=np.uint8).astype(np.int64)
    N, K2 = pk.shape
    K = 2 * K2
    codes = np.empty((N, K), dtype=np.int64)
    codes[:, 0::2] = pk & 0xF
    codes[:, 1::2] = pk >> 4
    sc = e4m3_value(np.asarray(scales, dtype=np.uint8))          # [K/16, N]
    blk = np.arange(K) // 16
    w = e2m1_value(codes) * sc[blk, :].T                          # [N, K]
    s2 = np.asarray(scale2, dtype=np.float32).astype(np.float64)
    if s2.ndim == 0:
        return w * s2
    return w * s2.reshape(-1, 1)


def dequant_fp8(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """FP8 (E4M3) weight of one expert -> fp64 ``W[n, kappa]``.

    The pages name FP8 grouped prefill weights beside NVFP4 and bf16 ([lora]
    module doc: the same fold serves the nvfp4, bf16 and fp8 grouped prefill
    paths) but print no layout. Reading, the plainest W8A16 one: E4M3 codes
    ``[N, K]`` (OCP FP8, bias 7, no infinities, 0x7F / 0xFF NaN), one fp32
    scale per output row, ``w[n, kappa] = e4m3(codes[n, kappa]) * scales[n]``.
    """
    v = e4m3_value(np.asarray(codes, dtype=np.uint8))                 # [N, K]
    s = np.asarray(scales, dtype=np.float32).astype(np.float64)
    return v * s.reshape(-1, 1)


def expert_weight(spec: dict, e: int) -> np.ndarray:
    """Dequantised fp64 ``W[n, kappa]`` of expert e for a weight spec.

    Spec dicts (stacked over experts, as the pages stack them):

    * ``{"format": "bf16", "w": uint16 [E, N, K]}``
    * ``{"format": "f64", "w": list of fp64 [N, K]}``: weights already expanded
      (e.g. by :func:`prepare_f64`), used as given
    * ``{"format": "gptq", "qweight": int32 [E, K/8, N], "scales": f16 [E, K/G, N],
      "qzeros": int32 [E, K/G, N/8], "group_size": G}``
    * ``{"format": "nvfp4", "packed": uint8 [E, N, K/2], "scales": uint8 [E, K/16, N],
      "scale2": f32 [S, E]}`` where ``S = 2`` for a gate/up weight (rows
      ``[0, N/2)`` take ``scale2[0, e]``, rows ``[N/2, N)`` take ``scale2[1, e]``)
      and ``S = 1`` otherwise.
    * ``{"format": "fp8", "codes": uint8 [E, N, K], "scales": f32 [E, N]}``
    """
    fmt = spec["format"]
    if fmt == "f64":
        return spec["w"][e]
    if fmt == "bf16":
        return dequant_bf16(spec["w"][e])
    if fmt == "gptq":
        return dequant_gptq(spec["qweight"][e], spec["scales"][e], spec["qzeros"][e],
                            int(spec["group_size"]))
    if fmt == "nvfp4":
        s2 = np.asarray(spec["scale2"], dtype=np.float32).reshape(-1, np.asarray(spec["packed"]).shape[0])
        N = np.asarray(spec["packed"]).shape[1]
        if s2.shape[0] == 2:
            row_s2 = np.where(np.arange(N) < N // 2, s2[0, e], s2[1, e])
        else:
            row_s2 = np.full(N, s2[0, e], dtype=np.float32)
        return dequant_nvfp4(spec["packed"][e], spec["scales"][e], row_s2)
    if fmt == "fp8":
        return dequant_fp8(spec["codes"][e], spec["scales"][e])
    raise ValueError(f"unknown weight format {fmt!r}")


def prepare_f64(spec: dict) -> dict:
    """Expand every expert of a weight spec to fp64 once (exact for every
    format), so repeated layer calls skip the per-call dequantisation."""
    E = next(v for k, v in spec.items() if k in ("w", "qweight", "packed", "codes")).__len__()
    return {"format": "f64", "w": [expert_weight(spec, e) for e in range(E)]}


# ----------------------------------------------------------------------------
# Steps a3 / a4: grouped gate/up (fused SiLU-mul) and grouped down GEMMs
# ----------------------------------------------------------------------------

def _expert_rows(offsets, sorted_ids, P, e, rows_subset):
    lo, hi = int(offsets[e]), int(offsets[e + 1])
    r = np.arange(lo, hi)
    r = r[np.asarray(sorted_ids)[r] != P]                # skip sentinel rows
    if rows_subset is not None:
        r = np.intersect1d(r, rows_subset)
    return r


def grouped_gate_up(x: np.ndarray, act: str, w_gate_up: dict, sorted_ids: np.ndarray,
                    expert_offsets: np.ndarray, P: int, top_k: int, inter: int,
                    rows_subset: Optional[np.ndarray] = None) -> np.ndarray:
    """Grouped gate/up GEMM with the SiLU-mul fused ([cutlass]
    ``nvfp4_grouped_gate_up_fused``; [triton] ``launch_fused_moe_w4a16_triton``;
    [lora] doc of ``moe_lora_grouped_down``: post-SiLU sorted activations).

    For every sorted row r of expert e holding pair p (not the sentinel), with
    token ``t = p // top_k``: ``g = x[t] . Wg_e^T`` and ``u = x[t] . Wu_e^T``
    (fp64 sums of exact products), where rows ``[0, I)`` of the stacked weight
    are the gate and rows ``[I, 2I)`` the up projection; then
    ``h[r] = act(silu(g) * u)`` with ``silu(g) = g / (1 + exp(-g))``.

    The result equals the per-expert dense GEMM on each expert's rows, which is
    how [cutlass] ``nvfp4_grouped_gate_up`` defines correctness. Returns fp64
    values (activation-rounded) ``[max_padded, I]``; rows not computed are NaN.
    """
    xs = act_to_f64(x, act)
    max_padded = np.asarray(sorted_ids).shape[0]
    h = np.full((max_padded, inter), np.nan)
    E = np.asarray(expert_offsets).shape[0] - 1
    for e in range(E):
        rows = _expert_rows(expert_offsets, sorted_ids, P, e, rows_subset)
        if rows.size == 0:
            continue
        W = expert_weight(w_gate_up, e)                      # [2I, H]
        tokens = np.asarray(sorted_ids)[rows] // top_k
        a = xs[tokens]
        g = a @ W[:inter].T
        u = a @ W[inter:2 * inter].T
        h[rows] = round_act(g / (1.0 + np.exp(-g)) * u, act)
    return h


def grouped_down(h: np.ndarray, act: str, w_down: dict, sorted_ids: np.ndarray,
                 expert_offsets: np.ndarray, P: int, hidden: int,
                 rows_subset: Optional[np.ndarray] = None) -> np.ndarray:
    """Grouped down GEMM ([cutlass] ``nvfp4_grouped_down``: the intermediate is
    already in expert order, no gather; writes ``c [M_total, N]``).

    ``y[r] = act(h[r] . Wd_e^T)`` for every non-sentinel row r of expert e
    (fp64 sums); ``h`` is fp64 values of activation-rounded numbers. Returns
    ``[max_padded, H]`` fp64, NaN where not computed.
    """
    max_padded = h.shape[0]
    y = np.full((max_padded, hidden), np.nan)
    E = np.asarray(expert_offsets).shape[0] - 1
    for e in range(E):
        rows = _expert_rows(expert_offsets, sorted_ids, P, e, rows_subset)
        if rows.size == 0:
            continue
        W = expert_weight(w_down, e)                         # [H, I]
        y[rows] = round_act(h[rows] @ W.T, act)
    return y


# ----------------------------------------------------------------------------
# Step a5: grouped LoRA shrink / expand fold
# ----------------------------------------------------------------------------

def lora_grouped_down(x: np.ndarray, base_out: np.ndarray, lora_a: dict, lora_b: dict,
                      scale: np.ndarray, n_experts: int, expert_offsets: np.ndarray,
                      sorted_ids: np.ndarray, P: int, top_k: int,
                      row_adapter: Optional[np.ndarray], row_offset: int, row_end: int,
                      x_gather: int = 0, xa: Optional[np.ndarray] = None):
    """Device-side grouped LoRA fold ([lora] ``moe_lora_grouped_down`` and
    ``MoeExpertRoute``), for one window ``[row_offset, row_end)`` of sorted rows.

    For expert ``e < n_experts`` with an adapter (``e in lora_a``), each row r of
    its span inside the window that holds a pair p (not the sentinel) and whose
    token ``p // top_k`` is adapted (``row_adapter`` is None, or
    ``row_adapter[token] >= 0``):

    * shrink: ``xa[r - row_offset, j] = bf16(sum_i x_row[i] * A_e[j, i])`` where
      ``x_row = x[r]`` (``x_gather = 0``, sorted activations) or
      ``x[p // top_k]`` (``x_gather = 1``, token-major input);
    * expand: ``delta[n] = bf16(sum_j xa[.., j] * B_e[n, j])``;
    * fold: ``base[r, n] = bf16(fp32(base[r, n]) + fp32(scale_e * fp32(delta[n])))``
      -- the page's ``base += scale * fp32(bf16(delta))`` with the multiply and
      the add each rounded to f32 (no fused multiply-add).

    ``A_e`` is ``[max_rank, k_in]`` and ``B_e`` is ``[n_out, max_rank]`` (the
    padded rank is B's row stride). All LoRA tensors are bf16 bit patterns;
    ``x`` and ``base_out`` are bf16 bits. Returns ``(new_base_bits, xa_bits)``;
    ``xa`` rows that no adapted row writes keep their input value (zeros if
    ``xa`` is None).
    """
    base = np.array(base_out, dtype=np.uint16, copy=True)
    xs = bf16_bits_to_f64(x)
    rank = next(iter(lora_a.values())).shape[0] if lora_a else 0
    window = max(0, row_end - row_offset)
    xa_out = (np.zeros((window, rank), dtype=np.uint16) if xa is None
              else np.array(xa, dtype=np.uint16, copy=True))
    for e in range(min(n_experts, np.asarray(expert_offsets).shape[0] - 1)):
        if e not in lora_a:
            continue
        lo = max(int(expert_offsets[e]), row_offset)
        hi = min(int(expert_offsets[e + 1]), row_end)
        A = bf16_bits_to_f64(lora_a[e])                      # [rank, k_in]
        B = bf16_bits_to_f64(lora_b[e])                      # [n_out, rank]
        s_e = np.float32(scale[e])
        for r in range(lo, hi):
            p = int(sorted_ids[r])
            if p == P:
                continue
            tok = p // top_k
            if row_adapter is not None and int(row_adapter[tok]) < 0:
                continue
            xr = xs[r] if x_gather == 0 else xs[tok]
            xa_row = round_to_bf16(A @ xr)                   # bf16 xa
            xa_out[r - row_offset] = f64_to_bf16_bits(xa_row)
            delta = round_to_bf16(B @ xa_row)                # bf16 delta
            prod = (np.float32(s_e) * delta.astype(np.float32)).astype(np.float32)
            acc = (bf16_bits_to_f64(base[r]).astype(np.float32) + prod).astype(np.float32)
            base[r] = f64_to_bf16_bits(acc.astype(np.float64))
    return base, xa_out


def lora_gather_bgmv(x: np.ndarray, base_out: np.ndarray, lora_a: dict, lora_b: dict,
                     scale: np.ndarray, n_experts: int, indices: np.ndarray, top_k: int,
                     row_adapter: Optional[np.ndarray], x_gather: int = 0,
                     xa: Optional[np.ndarray] = None):
    """Decode-path LoRA fold on slot-major rows ([lora] ``moe_lora_gather_bgmv``
    doc and launcher, ``gather_row_token``).

    The rows are the flat ``(token, slot)`` pairs ``s = t * top_k + j``, in that
    order, ``n_slots = indices.shape[0]`` of them (no expert sort, no padding).
    Row s takes its expert from ``indices[s]`` and its adapt decision from
    ``row_adapter[s // top_k]`` (``< 0``: the row is left alone; ``None``: every
    row folds). A row whose expert is ``>= n_experts`` or has no adapter is left
    alone too. The input row is ``x[s]`` (``x_gather = 0``: slot-major
    ``[n_slots, k_in]``, the down fold) or ``x[s // top_k]`` (``x_gather = 1``:
    token-major, the gate/up fold). Per folded row the arithmetic is that of
    :func:`lora_grouped_down`:

    * ``xa[s, j] = bf16(sum_i x_row[i] * A_e[j, i])``;
    * ``delta[n] = bf16(sum_j xa[s, j] * B_e[n, j])``;
    * ``base[s, n] = bf16(fp32(base[s, n]) + fp32(scale_e * fp32(delta[n])))``.

    Returns ``(new_base_bits, xa_bits)``; ``xa`` rows of rows left alone keep
    their input value (zeros if ``xa`` is None).
    """
    base = np.array(base_out, dtype=np.uint16, copy=True)
    xs = bf16_bits_to_f64(x)
    idx = np.asarray(indices).astype(np.int64)
    rank = next(iter(lora_a.values())).shape[0] if lora_a else 0
    xa_out = (np.zeros((idx.shape[0], rank), dtype=np.uint16) if xa is None
              else np.array(xa, dtype=np.uint16, copy=True))
    for s in range(idx.shape[0]):
        e = int(idx[s])
        if e >= n_experts or e not in lora_a:
            continue
        tok = s // top_k
        if row_adapter is not None and int(row_adapter[tok]) < 0:
            continue
        A = bf16_bits_to_f64(lora_a[e])                      # [rank, k_in]
        B = bf16_bits_to_f64(lora_b[e])                      # [n_out, rank]
        xr = xs[s] if x_gather == 0 else xs[tok]
        xa_row = round_to_bf16(A @ xr)
        xa_out[s] = f64_to_bf16_bits(xa_row)
        delta = round_to_bf16(B @ xa_row)
        prod = (np.float32(scale[e]) * delta.astype(np.float32)).astype(np.float32)
        acc = (bf16_bits_to_f64(base[s]).astype(np.float32) + prod).astype(np.float32)
        base[s] = f64_to_bf16_bits(acc.astype(np.float64))
    return base, xa_out


def gather_bgmv_grids(max_rank: int, n_out: int, n_slots: int):
    """The page's exact launch grids of the decode fold ([lora]
    ``gather_bgmv_grids``): ``([ceil(max_rank/4), n_slots, 1], [ceil(n_out/4),
    n_slots, 1])`` for the shrink and the expand, four outputs per 256-thread
    block. Kept as the record of the page's shape; the CUDA kernels size their
    own grids."""
    return ([-(-max_rank // 4), n_slots, 1], [-(-n_out // 4), n_slots, 1])


# ----------------------------------------------------------------------------
# Step a6: weighted top-k combine
# ----------------------------------------------------------------------------

def combine(y: np.ndarray, act: str, pair_to_row: np.ndarray, weights: np.ndarray,
            T: int, top_k: int, tokens: Optional[np.ndarray] = None) -> np.ndarray:
    """Weighted top-k combine ([ferrum] ``moe_combine``):
    ``out[t] = act(sum_j w[t, j] * y[pair_to_row[t*k + j]])`` (fp64 sum of the
    f32 weights times the activation-rounded expert outputs). Dropped pairs
    (``pair_to_row < 0``) contribute nothing. Returns fp64 ``[T, H]`` (or the
    listed ``tokens`` only, in that order)."""
    tokens = np.arange(T) if tokens is None else np.asarray(tokens)
    H = y.shape[1]
    out = np.zeros((tokens.shape[0], H))
    w = np.asarray(weights, dtype=np.float32).astype(np.float64).reshape(T, top_k)
    for i, t in enumerate(tokens):
        acc = np.zeros(H)
        for j in range(top_k):
            r = int(pair_to_row[t * top_k + j])
            if r >= 0:
                acc = acc + w[t, j] * y[r]
        out[i] = acc
    return round_act(out, act)


# ----------------------------------------------------------------------------
# The whole layer
# ----------------------------------------------------------------------------

@dataclass
class LayerResult:
    ids: np.ndarray
    weights: np.ndarray
    align: AlignResult
    h: np.ndarray
    y: np.ndarray          # after the LoRA fold when one is given
    out: np.ndarray        # [T or len(tokens), H]
    y_base: Optional[np.ndarray] = None   # before the fold (only with LoRA)


def moe_layer(x, act: str, logits, top_k: int, num_experts: int, block_size: int,
              w_gate_up: dict, w_down: dict, inter: int, hidden: int,
              renormalize: bool = True, lora: Optional[dict] = None,
              tokens: Optional[np.ndarray] = None, max_padded: Optional[int] = None
              ) -> LayerResult:
    """route -> align -> gate/up (+SiLU-mul) -> down (+ optional LoRA fold) -> combine.

    With ``tokens`` given, the FFN and the combine are evaluated only for the
    rows that belong to those tokens (routing and align always run in full);
    every other row of h, y is NaN and ``out`` holds the listed tokens only.
    ``lora`` (bf16 only): ``{"a": {e: [rank, I]}, "b": {e: [H, rank]},
    "scale": f32 [n_experts], "n_experts": n, "row_adapter": None or [T]}``.
    """
    T = np.asarray(logits).shape[0]
    ids, w = route_topk_softmax(logits, top_k, renormalize)
    P = T * top_k
    al = align_block_size(ids.reshape(-1), num_experts, block_size, max_padded)
    rows_subset = None
    if tokens is not None:
        pairs = (np.asarray(tokens)[:, None] * top_k + np.arange(top_k)[None, :]).reshape(-1)
        rows_subset = np.sort(al.pair_to_row[pairs])
    h = grouped_gate_up(x, act, w_gate_up, al.sorted_token_ids, al.expert_offsets, P,
                        top_k, inter, rows_subset)
    y = grouped_down(h, act, w_down, al.sorted_token_ids, al.expert_offsets, P, hidden,
                     rows_subset)
    y_base = None
    if lora is not None:
        if act != "bf16":
            raise ValueError("the LoRA fold is defined on bf16 activations")
        y_base = y
        rows = np.arange(y.shape[0]) if rows_subset is None else rows_subset
        h_bits = np.zeros(h.shape, dtype=np.uint16)
        y_bits = np.zeros(y.shape, dtype=np.uint16)
        h_bits[rows] = f64_to_bf16_bits(h[rows])
        y_bits[rows] = f64_to_bf16_bits(y[rows])
        sorted_for_fold = np.array(al.sorted_token_ids, copy=True)
        if rows_subset is not None:
            mask = np.ones(sorted_for_fold.shape[0], bool)
            mask[rows_subset] = False
            sorted_for_fold[mask] = P                      # untouched rows act as sentinels
        folded, _ = lora_grouped_down(h_bits, y_bits, lora["a"], lora["b"], lora["scale"],
                                      lora["n_experts"], al.expert_offsets, sorted_for_fold,
                                      P, top_k, lora.get("row_adapter"), 0, al.total_tokens_post_pad)
        y = np.full(y.shape, np.nan)
        y[rows] = bf16_bits_to_f64(folded[rows])
    out = combine(y, act, al.pair_to_row, w, T, top_k, tokens)
    return LayerResult(ids, w, al, h, y, out, y_base)
