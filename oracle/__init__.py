"""CPU oracle for the grouped mixture-of-experts expert-FFN path.

This package is TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it. The product path (the
CUDA library and its Python binding) never imports, links or runs anything here,
and nothing here imports the product package: the two share no code.

It is a plain, slow, obviously correct restatement of what the path computes,
written from the four source pages the method is taken from:

* ``spark_model/layers/ops/moe_lora_grouped.rs`` (Atlas inference docs): the
  grouped LoRA fold on the expert down projection;
* ``ferrum-kernels 0.7.7, src/backend/cuda/moe.rs``: top-k softmax routing,
  block-size alignment of (token, expert) pairs, the pair inverse map and the
  weighted combine;
* ``ferrum-kernels, src/backend/cuda/triton_fused_moe.rs``: the fused GPTQ
  INT4 x FP16 grouped GEMM (sorted_token_ids gather, expert_ids per block,
  sentinel rows, stacked raw GPTQ layout);
* ``metrale_gpu_runtime/cutlass/grouped.rs``: the grouped NVFP4 gate/up and
  down GEMMs and the ``ensure_group_arrays`` validation rules.

Floating point: every dot product is accumulated in fp64 (numpy ``matmul`` as
the library step). Values are rounded only where the pages store them in a
narrower type: router weights in f32, post-SiLU activations, expert outputs,
the LoRA ``xa`` and ``delta`` and the combined output in the activation dtype
(bf16 or fp16), and the LoRA ``base += scale * fp32(bf16(delta))`` step in f32.
"""

from .moe_oracle import *  # noqa: F401,F403
