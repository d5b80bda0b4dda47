"""Seeded synthetic inputs for the grouped MoE layer.

This module only draws random numbers and packs them into the storage formats
the layer consumes; it holds none of the layer's arithmetic. It imports neither
the CUDA binding nor the CPU oracle, and both the tests and ``bench.py`` feed
its output to each of them.

Every tensor draws from its own stream, ``PCG64(SeedSequence([seed, tensor,
expert]))``, so a weight does not depend on the token count and experts can be
drawn in parallel threads.

Workloads (names used across the tests and the benchmark):

* ``tiny``            T=16, H=128, I=64, E=8, k=2, bs=16, bf16
* ``mixtral_prefill`` T=4096, H=4096, I=14336, E=8, k=2, bs=64, bf16
* ``fine_grained``    H=2048, I=768, E=128, k=8, bs=64, bf16, Zipf-biased router
* ``gptq``            H=2048, I=1408, E=64, k=6, bs=16, fp16 activations, GPTQ int4
* ``nvfp4_lora``      T=2048, H=2048, I=768, E=128, k=8, bs=64, NVFP4 + rank-16 LoRA
* ``fp8``             T=2048, H=2048, I=768, E=128, k=8, bs=64, FP8 (E4M3) weights with
                      per-row fp32 scales, bf16 activations
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace
from typing import Optional

import numpy as np

# tensor stream ids
_X, _ROUTER, _GU, _DOWN, _LORA_A, _LORA_B, _GU_SC, _DOWN_SC, _S2 = range(9)


@dataclass(frozen=True)
class MoeConfig:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    bs: int
    act: str = "bf16"          # activation dtype: "bf16" | "f16"
    wfmt: str = "bf16"         # weight format: "bf16" | "gptq" | "nvfp4" | "fp8"
    router: str = "gemm"       # "gemm": logits = x @ Wr; "normal": N(0,1); "zipf": N(0,1) + bias
    router_std: float = 0.02   # std of Wr for router="gemm"
    weight_std: float = 0.02
    renormalize: bool = True
    lora_rank: int = 0         # 0 = no LoRA fold
    lora_scale: float = 2.0
    group_size: int = 128      # GPTQ group size
    nvfp4_recipe: str = "amax"  # NVFP4 weights: "amax" quantises a Gaussian, "draw" draws codes directly
    seed: int = 0

    def with_T(self, T: int) -> "MoeConfig":
        return replace(self, T=T, name=f"{self.name.split('@')[0]}@T{T}")

    @property
    def P(self) -> int:
        return self.T * self.k


CONFIGS = {
    "tiny": MoeConfig("tiny", T=16, H=128, I=64, E=8, k=2, bs=16, router_std=0.1),
    "mixtral_prefill": MoeConfig("mixtral_prefill", T=4096, H=4096, I=14336, E=8, k=2, bs=64,
                                 router_std=0.02),
    "fine_grained": MoeConfig("fine_grained", T=4096, H=2048, I=768, E=128, k=8, bs=64,
                              router="zipf"),
    "gptq": MoeConfig("gptq", T=2048, H=2048, I=1408, E=64, k=6, bs=16, act="f16",
                      wfmt="gptq", router="normal"),
    "nvfp4_lora": MoeConfig("nvfp4_lora", T=2048, H=2048, I=768, E=128, k=8, bs=64,
                            wfmt="nvfp4", router="normal", lora_rank=16),
    "fp8": MoeConfig("fp8", T=2048, H=2048, I=768, E=128, k=8, bs=64, wfmt="fp8", router="normal"),
}

FINE_GRAINED_T = (1, 8, 64, 512, 4096, 16384)
GPTQ_T = (16, 2048)


def _rng(seed: int, tensor: int, part: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tensor, part])))


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Pack f32 samples into bf16 storage (nearest, ties to even). Input packing
    only: finite samples from the generators below."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).copy()
    r = (u >> np.uint32(16)) & np.uint32(1)
    r += np.uint32(0x7FFF)
    u += r
    u >>= np.uint32(16)
    return u.astype(np.uint16)


def _normal_act(rng, shape, std, act):
    a = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return f32_to_bf16_bits(a) if act == "bf16" else a.astype(np.float16)


def _per_expert(fn, E):
    with ThreadPoolExecutor(_threads()) as ex:
        return np.stack(list(ex.map(fn, range(E))))


def _bf16_weight(seed, tensor, E, N, K, std):
    return {"format": "bf16",
            "w": _per_expert(lambda e: _normal_act(_rng(seed, tensor, e), (N, K), std, "bf16"), E)}


def _gptq_weight(seed, tensor, E, N, K, G):
    """Raw GPTQ layout: uniform 4-bit codes, fp16 scales U(0.005, 0.02), every
    zero point 8."""
    if K % 8 or K % G or N % 8:
        raise ValueError("GPTQ needs K % 8 == 0, K % group_size == 0, N % 8 == 0")

    def qw(e):
        return _rng(seed, tensor, e).integers(0, 2 ** 32, size=(K // 8, N), dtype=np.uint32).view(np.int32)

    def sc(e):
        return _rng(seed, tensor + 100, e).uniform(0.005, 0.02, size=(K // G, N)).astype(np.float16)

    zeros = np.full((E, K // G, N // 8), 0x88888888, dtype=np.uint32).view(np.int32)
    return {"format": "gptq", "qweight": _per_expert(qw, E), "scales": _per_expert(sc, E),
            "qzeros": zeros, "group_size": G}


# magnitude-code probabilities of E2M1 codes 0..7 (values 0,.5,1,1.5,2,3,4,6),
# shaped like a block-scaled Gaussian
_E2M1_P = np.array([0.10, 0.16, 0.18, 0.16, 0.14, 0.12, 0.09, 0.05])

# positive finite values of the two NVFP4 element formats in code order (OCP
# MX: E2M1 codes 0..7; E4M3 codes 0x00..0x7E, bias 7, subnormals m * 2^-9,
# 0x7F is NaN), the tables the quantising recipe rounds to
_E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
_E4M3_VALUES = np.array([m * 2.0 ** -9 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
                         for e in range(16) for m in range(8)][:127])


def _round_to_table(a: np.ndarray, table: np.ndarray) -> np.ndarray:
    """Codes of the nearest table values to a >= 0 (the table ascending in
    code order), ties to the even code, values past the largest saturating:
    round-to-nearest-even into a small float format."""
    a = np.minimum(a, table[-1])
    hi = np.clip(np.searchsorted(table, a, side="left"), 1, len(table) - 1)
    lo = hi - 1
    dlo = a - table[lo]
    dhi = table[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    return np.where(pick_hi, hi, lo).astype(np.uint8)


def _nvfp4_weight(seed, tensor, E, N, K, n_scale2, recipe="amax", std=0.02):
    """NVFP4 weights ([N, K/2] E2M1 codes, [K/16, N] E4M3 block scales, fp32
    scale2 [n_scale2, E]).

    ``amax`` (the default): block-amax quantisation of bf16 N(0, std) weights,
    per expert and per scale2 group (gate rows, up rows): scale2 = amax /
    (6 * 448); each 16-wide block's scale is the E4M3 rounding (nearest, ties
    to even) of amax_block / (6 * scale2); each weight's code is the E2M1
    rounding of w / (e4m3(scale) * scale2), saturating at 6. Every block then
    holds a code near +-6, as real quantised checkpoints do.

    ``draw``: codes drawn directly, E2M1 magnitude codes from ``_E2M1_P``
    with a random sign, E4M3 block scales with exponent field 5..9 and any
    mantissa (values 0.25 .. 3.75), scale2 U(0.5, 1.5) * 0.003: weights of
    RMS close to 0.02 that use every code and many scale values."""
    if K % 16:
        raise ValueError("NVFP4 needs K % 16 == 0")
    if recipe == "draw":
        def packed(e):
            r = _rng(seed, tensor, e)
            mag = r.choice(8, size=(N, K), p=_E2M1_P).astype(np.uint8)
            sign = r.integers(0, 2, size=(N, K), dtype=np.uint8) << 3
            c = mag | sign
            return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)

        def scales(e):
            r = _rng(seed, tensor + 100, e)
            ex = r.integers(5, 10, size=(K // 16, N), dtype=np.uint8)
            man = r.integers(0, 8, size=(K // 16, N), dtype=np.uint8)
            return ((ex << 3) | man).astype(np.uint8)

        s2 = (_rng(seed, _S2, tensor).uniform(0.5, 1.5, size=(n_scale2, E)) * 0.003).astype(np.float32)
        return {"format": "nvfp4", "packed": _per_expert(packed, E), "scales": _per_expert(scales, E),
                "scale2": s2}
    if recipe != "amax":
        raise ValueError(f"unknown NVFP4 recipe {recipe!r}")

    def quantise(e):
        bits = _normal_act(_rng(seed, tensor, e), (N, K), std, "bf16")
        w = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
        rows = N // n_scale2
        packed = np.empty((N, K // 2), np.uint8)
        sc = np.empty((K // 16, N), np.uint8)
        s2 = np.empty(n_scale2, np.float32)
        for g in range(n_scale2):
            wg = w[g * rows:(g + 1) * rows]
            amax = float(np.max(np.abs(wg)))
            s2g = np.float32(amax / (6.0 * 448.0)) if amax > 0 else np.float32(1.0)
            s2[g] = s2g
            blk = np.abs(wg).reshape(rows, K // 16, 16).max(axis=2)          # [rows, K/16]
            scode = _round_to_table(blk / (6.0 * float(s2g)), _E4M3_VALUES)   # [rows, K/16]
            sval = _E4M3_VALUES[scode] * float(s2g)
            denom = np.repeat(sval, 16, axis=1)
            mag = np.divide(np.abs(wg), denom, out=np.zeros_like(wg), where=denom > 0)
            c = _round_to_table(mag, _E2M1_VALUES) | (np.signbit(wg).astype(np.uint8) << 3)
            c = np.where(c == 8, 0, c).astype(np.uint8)                        # -0 as +0
            packed[g * rows:(g + 1) * rows] = c[:, 0::2] | (c[:, 1::2] << 4)
            sc[:, g * rows:(g + 1) * rows] = scode.T
        return packed, sc, s2

    with ThreadPoolExecutor(_threads()) as ex:
        parts = list(ex.map(quantise, range(E)))
    return {"format": "nvfp4", "packed": np.stack([p[0] for p in parts]),
            "scales": np.stack([p[1] for p in parts]),
            "scale2": np.ascontiguousarray(np.stack([p[2] for p in parts]).T)}


# E4M3 exponent-field probabilities (fields 0..10; 0 = zero and subnormals),
# so that most codes are 0.125 .. 7.5 and some are subnormal
_E4M3_EXP_P = np.array([0.03, 0.02, 0.03, 0.05, 0.09, 0.14, 0.18, 0.18, 0.14, 0.09, 0.05])


def _fp8_weight(seed, tensor, E, N, K):
    """FP8 (E4M3) codes drawn directly (random sign, exponent field from
    ``_E4M3_EXP_P``, any mantissa: never NaN) with one fp32 scale per output
    row U(0.5, 1.5) * 0.0075, so that the decoded weights have RMS close to
    0.02, the scale of the bf16 workloads."""
    def codes(e):
        r = _rng(seed, tensor, e)
        ex = r.choice(len(_E4M3_EXP_P), size=(N, K), p=_E4M3_EXP_P).astype(np.uint8)
        man = r.integers(0, 8, size=(N, K), dtype=np.uint8)
        sign = r.integers(0, 2, size=(N, K), dtype=np.uint8) << 7
        return (sign | (ex << 3) | man).astype(np.uint8)

    def scales(e):
        return (_rng(seed, tensor + 100, e).uniform(0.5, 1.5, size=N) * 0.0075).astype(np.float32)

    return {"format": "fp8", "codes": _per_expert(codes, E), "scales": _per_expert(scales, E)}


def make_weights(cfg: MoeConfig) -> dict:
    """Expert weights: gate/up stacked ``[E, 2I, H]`` (rows ``[0, I)`` gate,
    ``[I, 2I)`` up) and down ``[E, H, I]`` in the config's format."""
    E, H, I, s = cfg.E, cfg.H, cfg.I, cfg.seed
    if cfg.wfmt == "bf16":
        gu = _bf16_weight(s, _GU, E, 2 * I, H, cfg.weight_std)
        dn = _bf16_weight(s, _DOWN, E, H, I, cfg.weight_std)
    elif cfg.wfmt == "gptq":
        gu = _gptq_weight(s, _GU, E, 2 * I, H, cfg.group_size)
        dn = _gptq_weight(s, _DOWN, E, H, I, cfg.group_size)
    elif cfg.wfmt == "nvfp4":
        gu = _nvfp4_weight(s, _GU, E, 2 * I, H, 2, cfg.nvfp4_recipe, cfg.weight_std)
        dn = _nvfp4_weight(s, _DOWN, E, H, I, 1, cfg.nvfp4_recipe, cfg.weight_std)
    elif cfg.wfmt == "fp8":
        gu = _fp8_weight(s, _GU, E, 2 * I, H)
        dn = _fp8_weight(s, _DOWN, E, H, I)
    else:
        raise ValueError(cfg.wfmt)
    return {"w_gate_up": gu, "w_down": dn}


def make_lora(cfg: MoeConfig) -> Optional[dict]:
    """Rank-r bf16 LoRA on the down projection of the even-id experts:
    ``A_e [r, I]``, ``B_e [H, r]`` N(0, 0.02), scale ``cfg.lora_scale``; the
    tables run to the largest adapted id + 1."""
    if cfg.lora_rank == 0:
        return None
    adapted = list(range(0, cfg.E, 2))
    a = {e: _normal_act(_rng(cfg.seed, _LORA_A, e), (cfg.lora_rank, cfg.I), 0.02, "bf16") for e in adapted}
    b = {e: _normal_act(_rng(cfg.seed, _LORA_B, e), (cfg.H, cfg.lora_rank), 0.02, "bf16") for e in adapted}
    n = max(adapted) + 1
    scale = np.zeros(n, dtype=np.float32)
    scale[adapted] = np.float32(cfg.lora_scale)
    return {"a": a, "b": b, "scale": scale, "n_experts": n, "rank": cfg.lora_rank,
            "row_adapter": None}


def make_activations(cfg: MoeConfig) -> dict:
    """Token activations ``x [T, H]`` and router logits ``[T, E]`` (f32).

    * ``gemm``: ``Wr [H, E]`` f32 N(0, router_std) (returned as ``w_router``)
      and ``logits = f32(x @ Wr)`` with the product taken in fp64 (the router
      GEMM sits before the layer; its logits are part of the input recipe);
    * ``normal``: logits N(0, 1);
    * ``zipf``: logits N(0, 1) plus ``-1.1 * ln(e + 1)``, the log-probability of
      a Zipf(s=1.1) popularity with rank e + 1.
    """
    T, H, E, s = cfg.T, cfg.H, cfg.E, cfg.seed
    x = _normal_act(_rng(s, _X, T), (T, H), 1.0, cfg.act)
    r = _rng(s, _ROUTER, T)
    if cfg.router == "gemm":
        wr = _rng(s, _ROUTER, 0).standard_normal((H, E), dtype=np.float32) * np.float32(cfg.router_std)
        if cfg.act == "bf16":
            xf = (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
        else:
            xf = x.astype(np.float64)
        logits = (xf @ wr.astype(np.float64)).astype(np.float32)
        return {"x": x, "logits": logits, "w_router": wr}
    elif cfg.router == "normal":
        logits = r.standard_normal((T, E), dtype=np.float32)
    elif cfg.router == "zipf":
        bias = -1.1 * np.log(np.arange(E, dtype=np.float64) + 1.0)
        logits = (r.standard_normal((T, E)) + bias[None, :]).astype(np.float32)
    else:
        raise ValueError(cfg.router)
    return {"x": x, "logits": logits}


def make_inputs(cfg: MoeConfig, weights: Optional[dict] = None) -> dict:
    """Everything one layer call consumes, as numpy arrays."""
    d = make_activations(cfg)
    d.update(weights if weights is not None else make_weights(cfg))
    d["lora"] = make_lora(cfg)
    return d


def random_ids(seed: int, P: int, E: int, skew: float = 0.0) -> np.ndarray:
    """Flat expert ids for align tests: uniform, or Zipf-like with ``skew`` > 0."""
    r = _rng(seed, 50, P)
    if skew <= 0:
        return r.integers(0, E, size=P).astype(np.int32)
    p = (np.arange(E) + 1.0) ** -skew
    return r.choice(E, size=P, p=p / p.sum()).astype(np.int32)
