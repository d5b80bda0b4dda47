"""The align entry point for callers that cannot allocate device memory.

moe_align_block_size_noalloc keeps its scratch in a fixed array inside the
library instead of a caller-provided workspace. It exists for callers that
have no way to allocate device memory (a framework that owns the whole memory
budget and gives out no allocator, or a hot path that must not make an
allocation call, which can synchronise the device). These tests call it
through the C ABI twice in a row, with different shapes so that the second
call sees the first call's leftovers in the shared array, and check that its
outputs equal those of moe_align_block_size with a workspace (align is
compared bit for bit, as everywhere else). This file is collected last.
"""
import numpy as np
import pytest

from mixture_experts_grouped_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mixture_experts_grouped_gb300 import build
    build.build()
    return torch.device("cuda:0")


def _outputs(dev, P, E, bs):
    import torch
    from mixture_experts_grouped_gb300 import moe
    cap = moe.moe_align_capacity(P, E, bs)
    i32 = dict(dtype=torch.int32, device=dev)
    return dict(sorted=torch.full((cap,), -5, **i32), eids=torch.full((cap // bs,), -5, **i32),
                off=torch.full((E + 1,), -5, **i32), tot=torch.full((1,), -5, **i32),
                p2r=torch.full((max(P, 1),), -5, **i32), err=torch.zeros(1, **i32), cap=cap)


def _align_both(dev, ids_np, E, bs):
    import torch
    from mixture_experts_grouped_gb300 import moe
    P = ids_np.shape[0]
    ids = torch.from_numpy(ids_np.astype(np.int32)).to(dev)
    ref = _outputs(dev, P, E, bs)
    ws_bytes = moe.moe_align_workspace_size(P, E)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    moe.moe_align_block_size(ids, P, E, bs, ref["cap"], ref["sorted"], ref["eids"], ref["off"], ref["tot"],
                             ref["p2r"], ref["err"], ws, ws_bytes)
    got = _outputs(dev, P, E, bs)
    moe.moe_align_block_size_noalloc(ids, P, E, bs, got["cap"], got["sorted"], got["eids"], got["off"],
                                     got["tot"], got["p2r"], got["err"])
    torch.cuda.synchronize()
    return ref, got


def test_noalloc_align_matches_the_workspace_version_on_two_calls_in_a_row(dev):
    # first a large skewed routing, then a smaller one with other E / bs: the
    # second call runs on top of the first call's scratch contents
    cases = [(131072, 128, 64, 1.1), (3001, 16, 16, 0.0)]
    for P, E, bs, skew in cases:
        ids = synth.random_ids(7 * P + E, P, E, skew)
        ref, got = _align_both(dev, ids, E, bs)
        for key in ("sorted", "eids", "off", "tot", "p2r", "err"):
            assert np.array_equal(got[key].cpu().numpy(), ref[key].cpu().numpy()), (P, E, bs, key)
        assert int(got["err"].item()) == 0


def test_noalloc_rejects_more_pairs_than_its_scratch_holds(dev):
    import torch
    from mixture_experts_grouped_gb300 import moe
    P = moe.MOE_ALIGN_NOALLOC_MAX_PAIRS + 1
    i32 = dict(dtype=torch.int32, device=dev)
    buf = torch.zeros(8, **i32)
    n0 = moe.moe_launch_count()
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_align_block_size_noalloc(buf, P, 8, 16, moe.moe_align_capacity(P, 8, 16), buf, buf, buf, buf, buf,
                                         buf)
    assert ei.value.status == moe.MOE_ERR_INVALID and "fixed scratch" in ei.value.message
    assert moe.moe_launch_count() == n0
