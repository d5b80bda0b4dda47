"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, and its pure host logic follows the pages' rules."""
import json
import os
import re

import numpy as np
import pytest

import oracle as orc
from conftest import GOLDEN, ROOT


@pytest.fixture(scope="session")
def moe():
    from mixture_experts_grouped_gb300 import build as b
    b.build()
    from mixture_experts_grouped_gb300 import moe as m
    m.lib()
    return m


def header_functions():
    with open(os.path.join(ROOT, "include", "moe.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_six_path_calls():
    names = header_functions()
    for n in ["moe_route_topk_softmax", "moe_align_block_size", "moe_grouped_gate_up", "moe_grouped_down",
              "moe_lora_grouped_down", "moe_combine"]:
        assert n in names


def test_library_exports_every_declared_symbol(moe):
    lib = moe.lib()
    for name in header_functions():
        assert hasattr(lib, name), f"{name} declared in include/moe.h but not exported"
    # and the binding wraps each of them under the same name
    for name in header_functions():
        assert name in moe.exported_names() and hasattr(moe, name)


def test_group_array_vectors_through_the_abi(moe):
    with open(os.path.join(GOLDEN, "group_arrays_vectors.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        args = ("t", c["num_experts"], c["offsets"], [tuple(p) for p in c["per_expert"]])
        if c["ok"]:
            moe.moe_validate_group_arrays(*args)
        else:
            with pytest.raises(moe.MoeError) as ei:
                moe.moe_validate_group_arrays(*args)
            assert ei.value.status == moe.MOE_ERR_INVALID
            if "message_contains" in c:
                assert c["message_contains"] in ei.value.message


def test_capacity_matches_the_bound(moe):
    for P, E, bs in [(0, 8, 16), (1, 8, 16), (32, 8, 16), (8192, 8, 64), (131072, 128, 64), (12288, 64, 16),
                     (5, 300, 1)]:
        assert moe.moe_align_capacity(P, E, bs) == orc.align_capacity(P, E, bs)
    assert moe.moe_align_capacity(10, 8, 0) == -1
    assert moe.moe_align_capacity(-1, 8, 16) == -1


def test_workspace_sizes(moe):
    # the gathered rows (rounded up to 256 bytes), then the split-K area: 128 KB of
    # partial sums and 16 bytes of flags for each of 256 CTAs
    splitk = 256 * (128 * 1024 + 16)
    assert moe.moe_down_workspace_size() == splitk
    assert moe.moe_gate_up_workspace_size(8704, 4096) == 8704 * 4096 * 2 + splitk
    assert moe.moe_gate_up_workspace_size(3, 8) == 256 + splitk
    small = moe.moe_align_workspace_size(32, 8)
    big = moe.moe_align_workspace_size(131072, 128)
    assert small > 0 and big >= 131072 * 4 + 64 * 128 * 4


@pytest.mark.parametrize("call", [
    lambda m: m.moe_route_topk_softmax(0, 0, 0, 4, 300, 2, True, 0),            # E > MAX
    lambda m: m.moe_route_topk_softmax(0, 0, 0, 4, 8, 9, True, 0),              # top_k > E
    lambda m: m.moe_route_topk_softmax(0, 0, 0, 4, 64, 17, True, 0),            # top_k > MAX_TOPK
    lambda m: m.moe_router_topk_softmax(16, 0, 16, 4, 100, 8, 2, True, 16, 16, 16, 0),   # H % 8
    lambda m: m.moe_router_topk_softmax(16, 2, 16, 4, 128, 8, 2, True, 16, 16, 16, 0),   # act
    lambda m: m.moe_router_topk_softmax(16, 0, 16, 4, 128, 300, 2, True, 16, 16, 16, 0), # E > MAX
    lambda m: m.moe_router_topk_softmax(16, 0, None, 4, 128, 8, 2, True, 16, 16, 16, 0), # NULL weight
    lambda m: m.moe_route_topk_softmax(0, 0, 0, 4, 8, 2, True, 0),              # NULL pointers
    lambda m: m.moe_align_block_size(0, 32, 257, 16, 1024, 8, 8, 8, 8, 8, 0, 8, 1 << 20, 0),   # E > 256
    lambda m: m.moe_align_block_size(0, 32, 8, 0, 1024, 8, 8, 8, 8, 8, 0, 8, 1 << 20, 0),     # bs = 0
    lambda m: m.moe_align_block_size(16, 32, 8, 16, 144, 16, 16, 16, 16, 16, 0, 16, 1 << 20, 0),  # < capacity
    lambda m: m.moe_align_block_size(16, 32, 8, 16, 168, 16, 16, 16, 16, 16, 0, 16, 1 << 20, 0),  # not bs multiple
    lambda m: m.moe_align_block_size(16, 32, 8, 16, 160, 16, 16, 16, 16, 16, 0, 16, 4, 0),        # workspace small
    lambda m: m.moe_grouped_gate_up(16, 0, m.MoeWeight(0, 0, 16, None, None, None), 16, 16, 4, 2, 100, 64, 8,
                                    16, 64, 16, 0, 16, 1 << 30, 0),             # H % 8
    lambda m: m.moe_grouped_gate_up(16, 1, m.MoeWeight(0, 0, 16, None, None, None), 16, 16, 4, 2, 128, 64, 8,
                                    16, 64, 16, 0, 16, 1 << 30, 0),             # bf16 weight, f16 act
    lambda m: m.moe_grouped_gate_up(16, 1, m.MoeWeight(1, 100, 16, 16, 16, None), 16, 16, 4, 2, 128, 64, 8,
                                    16, 64, 16, 0, 16, 1 << 30, 0),             # GPTQ group not /64
    lambda m: m.moe_grouped_gate_up(16, 0, m.MoeWeight(7, 0, 16, None, None, None), 16, 16, 4, 2, 128, 64, 8,
                                    16, 64, 16, 0, 16, 1 << 30, 0),             # unknown format
    lambda m: m.moe_grouped_down(16, 0, m.MoeWeight(0, 0, 16, None, None, None), 16, 16, 4, 2, 128, 100, 8, 16, 64,
                                 16, 0, 16, 1 << 30, 0),                         # I % 8
    lambda m: m.moe_grouped_down(16, 0, m.MoeWeight(2, 0, 16, 16, None, 16), 16, 16, 4, 2, 128, 72, 8, 16, 64, 16,
                                 0, 16, 1 << 30, 0),                             # NVFP4 K % 32
    lambda m: m.moe_grouped_down(16, 1, m.MoeWeight(1, 64, 16, 16, 16, None), 16, 16, 4, 2, 200, 64, 8, 16, 64, 16,
                                 0, 16, 1 << 30, 0),                             # GPTQ H % 32
    lambda m: m.moe_combine(16, 0, 16, 16, 16, 4, 100, 2, 64, 0, 0),             # H % 8
    lambda m: m.moe_lora_grouped_down(m.MoeExpertRoute(16, 16, 16, 4, 64, 128, 65), 16, 16, 16, 16, None, 16,
                                      0, 64, 0, 8, 2, 0),                       # rank > MAX
    lambda m: m.moe_lora_grouped_down(m.MoeExpertRoute(16, 16, 16, 4, 64, 128, 16), 16, 16, 16, 16, None, 16,
                                      10, 5, 0, 8, 2, 0),                       # window reversed
    lambda m: m.moe_lora_gather_bgmv(m.MoeExpertRoute(16, 16, 16, 4, 64, 128, 65), 16, 16, 16, None, 16, 8, 2, 0, 0),
    lambda m: m.moe_lora_gather_bgmv(m.MoeExpertRoute(16, 16, 16, 4, 60, 128, 16), 16, 16, 16, None, 16, 8, 2, 0, 0),
    lambda m: m.moe_lora_gather_bgmv(m.MoeExpertRoute(16, 16, 16, 4, 64, 126, 16), 16, 16, 16, None, 16, 8, 2, 0, 0),
    lambda m: m.moe_lora_gather_bgmv(m.MoeExpertRoute(16, 16, 16, 4, 64, 128, 16), 16, 16, 16, None, 16, 8, 2, 2, 0),
    lambda m: m.moe_lora_gather_bgmv(m.MoeExpertRoute(16, 16, 16, 4, 64, 128, 16), 16, 16, 16, None, 16, 8, 0, 0, 0),
    lambda m: m.moe_lora_gather_bgmv(m.MoeExpertRoute(16, 16, 16, 4, 64, 128, 16), 16, 16, None, None, 16, 8, 2, 0, 0),
    lambda m: m.moe_lora_gather_bgmv(m.MoeExpertRoute(16, 16, 16, 4, 64, 128, 16), 24, 16, 16, None, 16, 8, 2, 0, 0),
])
def test_host_detected_misuse_returns_invalid_before_any_launch(moe, call):
    n0 = moe.moe_launch_count()
    with pytest.raises(moe.MoeError) as ei:
        call(moe)
    assert ei.value.status == moe.MOE_ERR_INVALID
    assert ei.value.message
    assert moe.moe_launch_count() == n0


def test_lora_host_helpers_follow_the_page(moe):
    with open(os.path.join(GOLDEN, "lora_window_math.json")) as f:
        g = json.load(f)
    for case in g["windows"]:
        assert moe.lora_windows(case["total"], case["cap"]) == [tuple(w) for w in case["windows"]]
    with pytest.raises(ValueError):
        moe.lora_windows(10, 0)
    for row, k, tok in g["row_token"]:
        assert row // k == tok
    assert moe.pack_expert_tables([]) is None
    a, b, s, n = moe.pack_expert_tables([(3, 10, 20, 0.5), (0, 1, 2, 2.0), (3, 11, 21, 0.25)])
    assert n == 4
    assert a == [1, 0, 0, 11] and b == [2, 0, 0, 21] and s == [2.0, 0.0, 0.0, 0.25]


def test_wait_limit_hook_returns_previous_and_restores_default(moe):
    """moe_set_wait_limit_ns (the GEMM kernels' wait limit, a testing hook)
    returns the previous limit; 0 restores the 2 s default. Host state only."""
    first = moe.moe_set_wait_limit_ns(12345)
    assert moe.moe_set_wait_limit_ns(0) == 12345
    assert moe.moe_set_wait_limit_ns(first) == 2_000_000_000
