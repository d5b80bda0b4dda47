"""ctypes binding of libmoe.so (declared in include/moe.h), same names as the C ABI.

Argument marshalling only: tensors become device pointers, a stream argument
of None means torch's current stream. Every call raises :class:`MoeError` on a
non-zero status with the library's message. The library must have been built
(``__graft_entry__.build()``); a missing library is an error, never a fallback.
"""

from __future__ import annotations

import ctypes
import os
import threading
from ctypes import c_char_p, c_int32, c_int64, c_size_t, c_uint32, c_uint64, c_void_p, POINTER

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe.so")

MOE_OK, MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA = 0, 1, 2, 3
MOE_DEV_ERR_EXPERT_ID, MOE_DEV_ERR_CAPACITY, MOE_DEV_ERR_OFFSETS, MOE_DEV_ERR_PAIR_ID, MOE_DEV_ERR_TIMEOUT = (
    0x1, 0x2, 0x4, 0x8, 0x10)
MOE_MAX_EXPERTS, MOE_MAX_TOPK, MOE_MAX_LORA_RANK = 256, 16, 64
MOE_ACT_BF16, MOE_ACT_F16 = 0, 1
MOE_W_BF16, MOE_W_GPTQ_INT4, MOE_W_NVFP4, MOE_W_FP8_E4M3 = 0, 1, 2, 3

ACT_CODES = {"bf16": MOE_ACT_BF16, "f16": MOE_ACT_F16}
WFMT_CODES = {"bf16": MOE_W_BF16, "gptq": MOE_W_GPTQ_INT4, "nvfp4": MOE_W_NVFP4, "fp8": MOE_W_FP8_E4M3}


class MoeError(RuntimeError):
    def __init__(self, name: str, status: int, message: str):
        super().__init__(f"{name} failed with status {status}: {message}")
        self.status = status
        self.message = message


class MoeWeight(ctypes.Structure):
    _fields_ = [("format", c_int32), ("group_size", c_int32), ("w", c_void_p), ("scales", c_void_p),
                ("zeros", c_void_p), ("scale2", c_void_p)]


class MoeExpertRoute(ctypes.Structure):
    _fields_ = [("a_table", c_void_p), ("b_table", c_void_p), ("scale_table", c_void_p), ("n_experts", c_uint32),
                ("k_in", c_uint32), ("n_out", c_uint32), ("max_rank", c_uint32)]


_SIGNATURES = {
    "moe_last_error": (c_char_p, []),
    "moe_launch_count": (c_uint64, []),
    "moe_set_wait_limit_ns": (c_uint64, [c_uint64]),
    "moe_route_topk_softmax": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32,
                                         c_void_p]),
    "moe_router_topk_softmax": (c_int32, [c_void_p, c_int32, c_void_p, c_int32, c_int32, c_int32, c_int32,
                                          c_int32, c_void_p, c_void_p, c_void_p, c_void_p]),
    "moe_align_capacity": (c_int64, [c_int64, c_int32, c_int32]),
    "moe_align_workspace_size": (c_size_t, [c_int32, c_int32]),
    "moe_align_block_size": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p,
                                       c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_align_block_size_noalloc": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_int32, c_void_p, c_void_p,
                                               c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "moe_gate_up_workspace_size": (c_size_t, [c_int32, c_int32]),
    "moe_grouped_gate_up": (c_int32, [c_void_p, c_int32, POINTER(MoeWeight), c_void_p, c_void_p, c_int32, c_int32,
                                      c_int32, c_int32, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p,
                                      c_size_t, c_void_p]),
    "moe_grouped_down": (c_int32, [c_void_p, c_int32, POINTER(MoeWeight), c_void_p, c_void_p, c_int32, c_int32,
                                   c_int32, c_int32, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p,
                                   c_size_t, c_void_p]),
    "moe_down_workspace_size": (c_size_t, []),
    "moe_lora_grouped_down": (c_int32, [POINTER(MoeExpertRoute), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                        c_void_p, c_uint32, c_uint32, c_uint32, c_int32, c_int32, c_void_p]),
    "moe_lora_gather_bgmv": (c_int32, [POINTER(MoeExpertRoute), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                       c_uint32, c_uint32, c_uint32, c_void_p]),
    "moe_combine": (c_int32, [c_void_p, c_int32, c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32,
                              c_void_p, c_void_p]),
    "moe_validate_group_arrays": (c_int32, [c_char_p, c_int32, POINTER(c_int32), c_int32, POINTER(c_char_p),
                                            POINTER(c_int32), c_int32]),
}

_lib = None
_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """Open libmoe.so once and declare its signatures."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                                       "(there is no fallback implementation)")
                handle = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in _SIGNATURES.items():
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = handle
    return _lib


def exported_names():
    return list(_SIGNATURES)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(name: str, rc: int) -> None:
    if rc != MOE_OK:
        raise MoeError(name, rc, lib().moe_last_error().decode(errors="replace"))


# ---- the C ABI, one wrapper per entry point --------------------------------------

def moe_last_error() -> str:
    return lib().moe_last_error().decode(errors="replace")


def moe_launch_count() -> int:
    return int(lib().moe_launch_count())


def moe_set_wait_limit_ns(ns: int) -> int:
    """Pipeline wait limit of later GEMM launches (0 = the 2 s default); returns the previous one."""
    return int(lib().moe_set_wait_limit_ns(int(ns)))


def moe_route_topk_softmax(logits, topk_ids, topk_weights, T, E, top_k, renormalize=True, stream=None):
    _check("moe_route_topk_softmax", lib().moe_route_topk_softmax(
        _ptr(logits), _ptr(topk_ids), _ptr(topk_weights), T, E, top_k, 1 if renormalize else 0, _stream(stream)))


def moe_router_topk_softmax(x, act, w_router, T, H, E, top_k, renormalize, logits, topk_ids, topk_weights,
                            stream=None):
    _check("moe_router_topk_softmax", lib().moe_router_topk_softmax(
        _ptr(x), act, _ptr(w_router), T, H, E, top_k, 1 if renormalize else 0, _ptr(logits), _ptr(topk_ids),
        _ptr(topk_weights), _stream(stream)))


def moe_align_capacity(P, E, block_size) -> int:
    return int(lib().moe_align_capacity(P, E, block_size))


def moe_align_workspace_size(P, E) -> int:
    return int(lib().moe_align_workspace_size(P, E))


def moe_align_block_size(topk_ids, P, E, block_size, max_padded, sorted_token_ids, expert_ids, expert_offsets,
                         total_tokens_post_pad, pair_to_row, err_word, workspace, workspace_bytes, stream=None):
    _check("moe_align_block_size", lib().moe_align_block_size(
        _ptr(topk_ids), P, E, block_size, max_padded, _ptr(sorted_token_ids), _ptr(expert_ids),
        _ptr(expert_offsets), _ptr(total_tokens_post_pad), _ptr(pair_to_row), _ptr(err_word), _ptr(workspace),
        workspace_bytes, _stream(stream)))


MOE_ALIGN_NOALLOC_MAX_PAIRS = 262144


def moe_align_block_size_noalloc(topk_ids, P, E, block_size, max_padded, sorted_token_ids, expert_ids,
                                 expert_offsets, total_tokens_post_pad, pair_to_row, err_word, stream=None):
    """moe_align_block_size for callers that cannot allocate device memory: the
    scratch is a fixed array inside the library (P <= 262144 pairs). Calls on
    one device share that array, so calls that overlap on the GPU race."""
    _check("moe_align_block_size_noalloc", lib().moe_align_block_size_noalloc(
        _ptr(topk_ids), P, E, block_size, max_padded, _ptr(sorted_token_ids), _ptr(expert_ids),
        _ptr(expert_offsets), _ptr(total_tokens_post_pad), _ptr(pair_to_row), _ptr(err_word), _stream(stream)))


def moe_gate_up_workspace_size(max_padded, H) -> int:
    return int(lib().moe_gate_up_workspace_size(max_padded, H))


def moe_grouped_gate_up(x, act, w_gate_up: MoeWeight, sorted_token_ids, expert_offsets, T, top_k, H, I, E,
                        block_size, max_padded, h_out, err_word, workspace, workspace_bytes, stream=None):
    _check("moe_grouped_gate_up", lib().moe_grouped_gate_up(
        _ptr(x), act, ctypes.byref(w_gate_up), _ptr(sorted_token_ids), _ptr(expert_offsets), T, top_k, H, I, E,
        block_size, max_padded, _ptr(h_out), _ptr(err_word), _ptr(workspace), workspace_bytes, _stream(stream)))


def moe_down_workspace_size() -> int:
    return int(lib().moe_down_workspace_size())


def moe_grouped_down(h, act, w_down: MoeWeight, sorted_token_ids, expert_offsets, T, top_k, H, I, E, block_size,
                     max_padded, y, err_word, workspace, workspace_bytes, stream=None):
    _check("moe_grouped_down", lib().moe_grouped_down(
        _ptr(h), act, ctypes.byref(w_down), _ptr(sorted_token_ids), _ptr(expert_offsets), T, top_k, H, I, E,
        block_size, max_padded, _ptr(y), _ptr(err_word), _ptr(workspace), workspace_bytes, _stream(stream)))


def moe_lora_gather_bgmv(route: MoeExpertRoute, x, base_out, indices, row_adapter, xa, n_slots, top_k, x_gather,
                         stream=None):
    _check("moe_lora_gather_bgmv", lib().moe_lora_gather_bgmv(
        ctypes.byref(route), _ptr(x), _ptr(base_out), _ptr(indices), _ptr(row_adapter), _ptr(xa), n_slots, top_k,
        x_gather, _stream(stream)))


def moe_lora_grouped_down(route: MoeExpertRoute, x, base_out, expert_offsets, sorted_token_ids, row_adapter, xa,
                          row_offset, row_end, x_gather, num_tokens, top_k, stream=None):
    _check("moe_lora_grouped_down", lib().moe_lora_grouped_down(
        ctypes.byref(route), _ptr(x), _ptr(base_out), _ptr(expert_offsets), _ptr(sorted_token_ids),
        _ptr(row_adapter), _ptr(xa), row_offset, row_end, x_gather, num_tokens, top_k, _stream(stream)))


def moe_combine(y, act, pair_to_row, topk_weights, out, T, H, top_k, max_padded, err_word=None, stream=None):
    _check("moe_combine", lib().moe_combine(
        _ptr(y), act, _ptr(pair_to_row), _ptr(topk_weights), _ptr(out), T, H, top_k, max_padded, _ptr(err_word),
        _stream(stream)))


def moe_validate_group_arrays(who: str, num_experts: int, offsets, per_expert) -> None:
    """Host-side check of a grouped launch's arrays (no GPU needed).
    ``per_expert`` is a list of ``(name, length)``."""
    offs = (c_int32 * max(1, len(offsets)))(*[int(o) for o in offsets])
    names = (c_char_p * max(1, len(per_expert)))(*[n.encode() for n, _ in per_expert])
    lens = (c_int32 * max(1, len(per_expert)))(*[int(n) for _, n in per_expert])
    _check("moe_validate_group_arrays", lib().moe_validate_group_arrays(
        who.encode(), num_experts, offs, len(offsets), names, lens, len(per_expert)))


# ---- pure host helpers of the LoRA launcher (no GPU) -------------------------------

def pack_expert_tables(entries):
    """Dense per-expert LoRA tables from ``(expert_id, a_addr, b_addr, scale)``
    entries (spark_model moe_lora_grouped.rs, pack_expert_tables): ``None`` for
    no entries; ``n_experts = max id + 1``; unadapted slots hold 0 / 0.0; a
    repeated id keeps its last entry. Returns ``(a, b, scale, n_experts)``."""
    if not entries:
        return None
    n = max(int(e) for e, *_ in entries) + 1
    a, b, s = [0] * n, [0] * n, [0.0] * n
    for e, a_addr, b_addr, sc in entries:
        a[int(e)], b[int(e)], s[int(e)] = int(a_addr), int(b_addr), float(sc)
    return a, b, s, n


def lora_windows(total_rows: int, cap: int):
    """Contiguous ``[start, end)`` windows of at most ``cap`` rows covering
    ``[0, total_rows)`` (spark_model moe_lora_grouped.rs,
    grouped_down_windows); ``cap`` must be positive."""
    if cap <= 0:
        raise ValueError("grouped LoRA scratch capacity must be nonzero")
    return [(s, min(s + cap, total_rows)) for s in range(0, total_rows, cap)]
