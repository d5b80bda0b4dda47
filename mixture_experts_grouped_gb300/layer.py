"""One MoE layer on the GPU through the C ABI: device buffers and the call sequence.

PyTorch only provides device memory and the stream; every step runs in
libmoe.so. The sequence is route -> align -> gate/up (+SiLU-mul) -> down ->
optional LoRA fold -> combine, all enqueued on one stream with no host
synchronisation, so :meth:`MoeLayer.forward` can be captured in a CUDA graph.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

from . import moe as M


def act_dtype(act: str) -> torch.dtype:
    return torch.bfloat16 if act == "bf16" else torch.float16


def act_tensor(a: np.ndarray, act: str, device) -> torch.Tensor:
    """Activation storage from numpy (uint16 bf16 bits or float16) to a device tensor."""
    if act == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float16))
    return t.to(device)


def act_numpy(t: torch.Tensor, act: str) -> np.ndarray:
    """Device activation tensor back to numpy storage (uint16 bits or float16)."""
    t = t.detach().cpu()
    if act == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


@dataclass
class DeviceWeight:
    desc: M.MoeWeight
    tensors: list = field(default_factory=list)  # keeps the device memory alive

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in self.tensors)


def upload_weight(spec: dict, act: str, device) -> DeviceWeight:
    """A stacked weight spec (see oracle / synth conventions) to device memory."""
    fmt = spec["format"]
    if fmt == "bf16":
        w = act_tensor(spec["w"], "bf16", device)
        return DeviceWeight(M.MoeWeight(M.MOE_W_BF16, 0, w.data_ptr(), None, None, None), [w])
    if fmt == "gptq":
        qw = torch.from_numpy(np.ascontiguousarray(spec["qweight"])).to(device)
        sc = torch.from_numpy(np.ascontiguousarray(spec["scales"], dtype=np.float16)).to(device)
        qz = torch.from_numpy(np.ascontiguousarray(spec["qzeros"])).to(device)
        return DeviceWeight(M.MoeWeight(M.MOE_W_GPTQ_INT4, int(spec["group_size"]), qw.data_ptr(), sc.data_ptr(),
                                        qz.data_ptr(), None), [qw, sc, qz])
    if fmt == "nvfp4":
        pk = torch.from_numpy(np.ascontiguousarray(spec["packed"])).to(device)
        sc = torch.from_numpy(np.ascontiguousarray(spec["scales"])).to(device)
        s2 = torch.from_numpy(np.ascontiguousarray(spec["scale2"], dtype=np.float32)).to(device)
        return DeviceWeight(M.MoeWeight(M.MOE_W_NVFP4, 0, pk.data_ptr(), sc.data_ptr(), None, s2.data_ptr()),
                            [pk, sc, s2])
    if fmt == "fp8":
        cd = torch.from_numpy(np.ascontiguousarray(spec["codes"])).to(device)
        sc = torch.from_numpy(np.ascontiguousarray(spec["scales"], dtype=np.float32)).to(device)
        return DeviceWeight(M.MoeWeight(M.MOE_W_FP8_E4M3, 0, cd.data_ptr(), sc.data_ptr(), None, None), [cd, sc])
    raise ValueError(f"unknown weight format {fmt!r}")


@dataclass
class DeviceLora:
    route: M.MoeExpertRoute
    tensors: list


def upload_lora(lora: dict, k_in: int, n_out: int, device) -> DeviceLora:
    """Per-expert A_e / B_e to device plus the dense address / scale tables."""
    keep = []
    entries = []
    for e, a in lora["a"].items():
        ta = act_tensor(a, "bf16", device)
        tb = act_tensor(lora["b"][e], "bf16", device)
        keep += [ta, tb]
        entries.append((e, ta.data_ptr(), tb.data_ptr(), float(lora["scale"][e])))
    a_tab, b_tab, s_tab, n = M.pack_expert_tables(entries)
    at = torch.tensor(np.array(a_tab, dtype=np.uint64).view(np.int64), device=device)
    bt = torch.tensor(np.array(b_tab, dtype=np.uint64).view(np.int64), device=device)
    st = torch.tensor(np.array(s_tab, dtype=np.float32), device=device)
    keep += [at, bt, st]
    route = M.MoeExpertRoute(at.data_ptr(), bt.data_ptr(), st.data_ptr(), n, k_in, n_out, int(lora["rank"]))
    return DeviceLora(route, keep)


class MoeLayer:
    """Buffers for one (T, H, I, E, k, bs) shape and the five/six ABI calls."""

    def __init__(self, T, H, I, E, k, bs, act, w_gate_up: DeviceWeight, w_down: DeviceWeight, device="cuda",
                 lora: Optional[DeviceLora] = None, renormalize: bool = True, row_adapter=None):
        self.T, self.H, self.I, self.E, self.k, self.bs = T, H, I, E, k, bs
        self.act, self.act_code = act, M.ACT_CODES[act]
        self.P = T * k
        self.w_gate_up, self.w_down, self.lora = w_gate_up, w_down, lora
        self.renormalize = renormalize
        self.row_adapter = row_adapter
        self.max_padded = M.moe_align_capacity(self.P, E, bs)
        i32 = dict(dtype=torch.int32, device=device)
        dt = act_dtype(act)
        self.topk_ids = torch.empty((T, k), **i32)
        self.topk_weights = torch.empty((T, k), dtype=torch.float32, device=device)
        self.sorted_token_ids = torch.empty(self.max_padded, **i32)
        self.expert_ids = torch.empty(max(1, self.max_padded // bs), **i32)
        self.expert_offsets = torch.empty(E + 1, **i32)
        self.total_post_pad = torch.empty(1, **i32)
        self.pair_to_row = torch.empty(max(1, self.P), **i32)
        self.err = torch.zeros(1, **i32)
        self.align_ws_bytes = M.moe_align_workspace_size(self.P, E)
        self.align_ws = torch.empty(self.align_ws_bytes, dtype=torch.uint8, device=device)
        self.gate_up_ws_bytes = M.moe_gate_up_workspace_size(self.max_padded, H)
        # zeroed: both GEMM workspaces end in a split-K area that must start at zero
        self.gate_up_ws = torch.zeros(max(1, self.gate_up_ws_bytes), dtype=torch.uint8, device=device)
        self.down_ws_bytes = M.moe_down_workspace_size()
        self.down_ws = torch.zeros(self.down_ws_bytes, dtype=torch.uint8, device=device)
        self.h = torch.empty((self.max_padded, I), dtype=dt, device=device)
        self.y = torch.empty((self.max_padded, H), dtype=dt, device=device)
        self.out = torch.empty((T, H), dtype=dt, device=device)
        self.xa = (torch.empty((self.max_padded, lora.route.max_rank), dtype=torch.bfloat16, device=device)
                   if lora is not None else None)

    # individual steps ------------------------------------------------------------
    def route(self, logits, stream=None):
        M.moe_route_topk_softmax(logits, self.topk_ids, self.topk_weights, self.T, self.E, self.k,
                                 self.renormalize, stream)

    def align(self, stream=None):
        M.moe_align_block_size(self.topk_ids, self.P, self.E, self.bs, self.max_padded, self.sorted_token_ids,
                               self.expert_ids, self.expert_offsets, self.total_post_pad, self.pair_to_row,
                               self.err, self.align_ws, self.align_ws_bytes, stream)

    def gate_up(self, x, stream=None):
        M.moe_grouped_gate_up(x, self.act_code, self.w_gate_up.desc, self.sorted_token_ids, self.expert_offsets,
                              self.T, self.k, self.H, self.I, self.E, self.bs, self.max_padded, self.h, self.err,
                              self.gate_up_ws, self.gate_up_ws_bytes, stream)

    def down(self, stream=None):
        M.moe_grouped_down(self.h, self.act_code, self.w_down.desc, self.sorted_token_ids, self.expert_offsets,
                           self.T, self.k, self.H, self.I, self.E, self.bs, self.max_padded, self.y, self.err,
                           self.down_ws, self.down_ws_bytes, stream)

    def lora_fold(self, stream=None, row_offset=0, row_end=None):
        if self.lora is None:
            return
        end = self.max_padded if row_end is None else row_end
        M.moe_lora_grouped_down(self.lora.route, self.h, self.y, self.expert_offsets, self.sorted_token_ids,
                                self.row_adapter, self.xa, row_offset, end, 0, self.T, self.k, stream)

    def combine(self, stream=None):
        M.moe_combine(self.y, self.act_code, self.pair_to_row, self.topk_weights, self.out, self.T, self.H, self.k,
                      self.max_padded, self.err, stream)

    def forward(self, x, logits, stream=None):
        """The whole layer; returns the output tensor [T, H] (written in place)."""
        self.route(logits, stream)
        self.align(stream)
        self.gate_up(x, stream)
        self.down(stream)
        self.lora_fold(stream)
        self.combine(stream)
        return self.out

    def capture(self, x, logits):
        """CUDA graphs of one forward: (pre = route + align, gate_up, post =
        down + fold + combine) and the whole layer. The buffers are fixed, so
        replaying a graph re-runs the layer on the current contents of x and
        logits. Returns (pre, gate_up, post, whole, kernels_per_forward)."""
        self.forward(x, logits)          # first use on this device (attributes, descriptors)
        torch.cuda.synchronize()
        graphs = []
        n0 = M.moe_launch_count()
        for part in ("pre", "gate_up", "post"):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                if part == "pre":
                    self.route(logits)
                    self.align()
                elif part == "gate_up":
                    self.gate_up(x)
                else:
                    self.down()
                    self.lora_fold()
                    self.combine()
            graphs.append(g)
        per_forward = M.moe_launch_count() - n0
        whole = torch.cuda.CUDAGraph()
        with torch.cuda.graph(whole):
            self.forward(x, logits)
        torch.cuda.synchronize()
        return graphs[0], graphs[1], graphs[2], whole, per_forward

    @property
    def launches_per_forward(self) -> int:
        align = 1 if self.P <= 2048 else 3
        return 1 + align + 2 + 1 + (2 if self.lora is not None else 0) + 1
