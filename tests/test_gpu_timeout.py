"""A pipeline wait that runs out ends the GEMM cleanly, with an error status.

Every mbarrier and split-K flag wait inside the grouped GEMM kernels is
bounded. When one runs out, the kernel records MOE_DEV_ERR_TIMEOUT in the
call's error word, lets the copies and MMAs it has in flight land, frees its
tensor memory and returns: the error model of the pages is a status return
(metrale_gpu_runtime/cutlass/grouped.rs, a C status != 0 becomes an error),
never a trap. These tests set the limit to a few hundred nanoseconds through
the library's testing hook (moe_set_wait_limit_ns), so that the first waits
of the decode form (bf16 weights, with and without tiles cut across CTAs) and
of the TS form (quantised weights) give up, and then check that

  * the calls return (the kernels ended) with the timeout bit set;
  * the context stays usable: the next layer at the default limit, with the
    split-K areas left as the timed-out calls left them (their flags carry an
    older call's generation, which no later call accepts), finishes without a
    device error and its outputs are bit-identical to those of a clean run
    before the timeout.

Nothing here faults, traps or waits on a flag that is never set: the waits
themselves are ordinary pipeline waits that would complete a microsecond
later.
"""
import pytest

from mixture_experts_grouped_gb300 import synth
from parity import gpu_layer

pytestmark = pytest.mark.gpu

CASES = {
    # bf16 decode form; fewer tiles than SMs, so tiles are cut into k pieces
    # and the owner CTAs wait on their peers' split-K flags
    "decode_splitk": synth.MoeConfig("decode_splitk", T=6, H=1000, I=520, E=4, k=2, bs=16, router="normal"),
    # bf16 decode form with whole tiles (fine-grained layer, 64 tokens)
    "decode_fine_grained_T64": synth.CONFIGS["fine_grained"].with_T(64),
    # TS form: GPTQ int4 weights, fp16 activations, two sets of dequantising warps
    "ts_gptq_T16": synth.CONFIGS["gptq"].with_T(16),
    # TS form: FP8 weights, one set of dequantising warps
    "ts_fp8_decode": synth.MoeConfig("ts_fp8_decode", T=24, H=272, I=144, E=8, k=2, bs=16, wfmt="fp8",
                                     router="normal"),
}


@pytest.fixture(scope="module")
def dev():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mixture_experts_grouped_gb300 import build
    build.build()
    return torch.device("cuda:0")


@pytest.mark.parametrize("name", list(CASES))
def test_wait_timeout_returns_and_context_recovers(dev, name):
    import torch
    from mixture_experts_grouped_gb300 import moe
    cfg = CASES[name]
    inp = synth.make_inputs(cfg)
    lay, x, logits = gpu_layer(cfg, inp, dev)
    assert int(lay.err.item()) == 0
    clean = [t.clone() for t in (lay.h, lay.y, lay.out)]

    prev = moe.moe_set_wait_limit_ns(300)
    try:
        lay.err.zero_()
        lay.gate_up(x)      # both calls return MOE_OK (the binding raises otherwise) ...
        lay.down()
        torch.cuda.synchronize()  # ... and their kernels end
        err = int(lay.err.item())
    finally:
        moe.moe_set_wait_limit_ns(prev)
    assert err & moe.MOE_DEV_ERR_TIMEOUT, f"no wait ran out: error word {err:#x}"
    assert err & ~moe.MOE_DEV_ERR_TIMEOUT == 0, f"unexpected error bits {err:#x}"

    # nothing to clean up but the error word: the split-K areas stay as they are
    lay.err.zero_()
    lay.forward(x, logits)
    torch.cuda.synchronize()
    assert int(lay.err.item()) == 0
    for what, a, b in zip(("h", "y", "out"), clean, (lay.h, lay.y, lay.out)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"{what} differs from the clean run"
    # and the split-K flags are left zero again
    assert not lay.gate_up_ws[-4096:].any() and not lay.down_ws[-4096:].any()

