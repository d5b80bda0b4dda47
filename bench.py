#!/usr/bin/env python3
"""Throughput of the grouped MoE layer on GB300, one JSON line on rank 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the whole hot path over one batch: route -> align ->
gate/up (+SiLU-mul) -> down -> (LoRA fold) -> combine, through the C ABI, with
inputs and weights resident in HBM. The default workload is the Mixtral-style
prefill layer (T=4096, H=4096, I=14336, E=8, top_k=2, block_size=64, bf16).
Its 2.8 GB of expert weights stream from HBM every step, far more than the
126 MB L2, so no L2 flush is needed between steps.

Under torchrun (N > 1) every rank runs an independent replica of the layer on
its own GPU (no data-path collective); the timed region is bracketed by
barriers and the max over ranks is reported (weak scaling).

--impl reference times the CPU oracle (plain numpy, fp64) on the host cores,
each step a small sub-batch of the same workload.

Two single-call micro-benchmarks print their own JSON line instead:
--fold-only times the decode LoRA fold (moe_lora_gather_bgmv) on the
workload's slot-major rows, --router-only the router GEMM + routing
(moe_router_topk_softmax) on a workload with a router weight.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s and TFLOP/s or weight GB/s vs GB300 roofline, 1 GPU"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=600)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="mixtral_prefill")
    ap.add_argument("--override", default="", help="comma-separated field=value changes, e.g. E=2,T=1024")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU-baseline time budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--router-only", action="store_true",
                    help="time the router GEMM + routing (moe_router_topk_softmax) alone on the workload's tokens")
    ap.add_argument("--fold-only", action="store_true",
                    help="time the decode LoRA fold (moe_lora_gather_bgmv) alone on the workload's slot-major rows")
    a = ap.parse_args()
    if a.warmup < 3:
        ap.error("--warmup must be at least 3")
    return a


def workload(name):
    from mixture_experts_grouped_gb300 import synth
    if "@T" in name:
        base, t = name.split("@T")
        return synth.CONFIGS[base].with_T(int(t))
    return synth.CONFIGS[name]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def algorithmic(cfg, ids):
    """FLOPs of the two GEMMs (padding excluded) and bytes of the experts the
    routing touched (weights incl. scales / zeros) plus activation traffic."""
    import numpy as np
    P, H, I = cfg.P, cfg.H, cfg.I
    flops_gate_up = 2.0 * P * H * 2 * I
    flops_down = 2.0 * P * I * H
    touched = int(np.unique(ids).shape[0])
    if cfg.wfmt == "bf16":
        per_expert = (2 * I * H + H * I) * 2
    elif cfg.wfmt == "gptq":
        G = cfg.group_size
        per_expert = sum(K * N // 2 + (K // G) * N * 2 + (K // G) * (N // 8) * 4 for K, N in ((H, 2 * I), (I, H)))
    elif cfg.wfmt == "fp8":
        per_expert = sum(K * N + N * 4 for K, N in ((H, 2 * I), (I, H)))
    else:
        per_expert = sum(K * N // 2 + (K // 16) * N + 4 for K, N in ((H, 2 * I), (I, H)))
    act = 2
    act_bytes = (cfg.T * H * act          # x read (gather)
                 + P * H * act * 2        # gathered rows written + read by the GEMM
                 + P * I * act * 2        # h written + read
                 + P * H * act * 2        # y written + read
                 + cfg.T * H * act)       # out written
    if cfg.wfmt == "bf16":
        gu_weight = 2 * I * H * 2
    elif cfg.wfmt == "gptq":
        G = cfg.group_size
        gu_weight = H * 2 * I // 2 + (H // G) * 2 * I * 2 + (H // G) * (2 * I // 8) * 4
    elif cfg.wfmt == "fp8":
        gu_weight = H * 2 * I + 2 * I * 4
    else:
        gu_weight = H * 2 * I // 2 + (H // 16) * 2 * I + 8
    # the gate/up call: gather (x read, rows written), GEMM (rows read, weights, h written)
    gu_bytes = touched * gu_weight + cfg.T * H * act + 2 * P * H * act + P * I * act
    return {"flops_gate_up": flops_gate_up, "flops_down": flops_down, "flops": flops_gate_up + flops_down,
            "touched_experts": touched, "weight_bytes": touched * per_expert,
            "bytes": touched * per_expert + act_bytes, "gate_up_bytes": gu_bytes}


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                pw.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm_sorted = sorted(sm)
        return {"sm_mhz": sm_sorted[len(sm_sorted) // 2], "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(pw)}


def tensor_peak(pk: dict, clk: dict):
    """The bf16 tensor peak a kernel timed in this run is held to: the burst
    figure (a matmul timed alone at full clocks) unless the clocks sampled
    during the timed region show the power cap, or a median SM clock below
    97% of the maximum, in which case the sustained figure (a seconds-long
    matmul loop under the power cap). Returns (TFLOP/s, which)."""
    burst = float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sustained = float(pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    sm, mx = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    capped = "sw_power_cap" in clk.get("reasons", []) or (sm is not None and mx and sm < 0.97 * mx)
    return (sustained, "sustained") if capped else (burst, "burst")


def traffic_for(kernel_key: str, workload: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, valid only for the workload it was captured on and while the
    kernel source is the one that was profiled."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f).get(kernel_key)
    except (OSError, ValueError):
        return None
    if not d or d.get("workload") != workload:
        return None
    src = os.path.join(ROOT, d["source"])
    try:
        with open(src, "rb") as f:
            h = hashlib.sha256(f.read()).hexdigest()[:16]
    except OSError:
        return None
    return d["bytes_per_launch"] if h == d["source_sha256_16"] else None


# ----------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and the reference arm)
# ----------------------------------------------------------------------------

def oracle_setup(cfg, inp=None):
    import oracle as orc
    from mixture_experts_grouped_gb300 import synth
    if inp is None:
        inp = synth.make_inputs(cfg)
    wgu = orc.prepare_f64(inp["w_gate_up"])
    wd = orc.prepare_f64(inp["w_down"])
    return inp, wgu, wd


def oracle_step(cfg, inp, wgu, wd, t0, n_tok):
    """The whole oracle layer on tokens [t0, t0 + n_tok) of the workload."""
    import oracle as orc
    x = inp["x"][t0:t0 + n_tok]
    lg = inp["logits"][t0:t0 + n_tok]
    return orc.moe_layer(x, cfg.act, lg, cfg.k, cfg.E, cfg.bs, wgu, wd, cfg.I, cfg.H, cfg.renormalize,
                         lora=inp["lora"])


def oracle_threads():
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 0) for i in threadpool_info()), default=0)
        if n:
            return n
    except ImportError:
        pass
    return os.cpu_count() or 1


def cpu_baseline(cfg, budget_s, inp=None):
    inp, wgu, wd = oracle_setup(cfg, inp)
    n_tok = 32 if cfg.T >= 32 else cfg.T
    oracle_step(cfg, inp, wgu, wd, 0, n_tok)          # untimed warm-up
    done, t_start, reps = 0, time.perf_counter(), 0
    while True:
        t0 = (reps * n_tok) % max(1, cfg.T - n_tok + 1)
        oracle_step(cfg, inp, wgu, wd, t0, n_tok)
        done += n_tok
        reps += 1
        el = time.perf_counter() - t_start
        if el >= budget_s or reps >= 10000:
            break
    return {"value": done / el, "unit": "tokens/s", "cores": oracle_threads(), "kind": "oracle",
            "sample": f"{reps} sub-batches of {n_tok} consecutive tokens of the {cfg.name} workload "
                      f"(whole layer per sub-batch, fp64 weights expanded before timing), {el:.1f} s"}


def run_reference(args, cfg, rank, world):
    base = {"impl": "reference", "metric": METRIC, "unit": "tokens/s", "higher_is_better": True,
            "n_gpus": world, "scaling": "weak"}
    if rank != 0:
        return None
    inp, wgu, wd = oracle_setup(cfg)
    # size each step's sub-batch so that the whole run ends within about two minutes
    t = time.perf_counter()
    oracle_step(cfg, inp, wgu, wd, 0, 1)
    per_token = max(time.perf_counter() - t, 1e-4)
    n_tok = int(max(1, min(cfg.T, 120.0 / (per_token * (args.steps + args.warmup)))))
    for i in range(args.warmup):
        oracle_step(cfg, inp, wgu, wd, (i * n_tok) % max(1, cfg.T - n_tok + 1), n_tok)
    t = time.perf_counter()
    for i in range(args.steps):
        oracle_step(cfg, inp, wgu, wd, (i * n_tok) % max(1, cfg.T - n_tok + 1), n_tok)
    el = time.perf_counter() - t
    value = args.steps * n_tok / el
    sample = (f"each step the whole oracle layer on {n_tok} consecutive tokens of the {cfg.name} workload "
              f"(fp64 weights expanded before timing)")
    base.update({"value": value, "steps": args.steps, "warmup": args.warmup,
                 "ms_per_step": 1e3 * el / args.steps, "vs_baseline": None, "dtype": "f64",
                 "data": "synthetic (seeded)", "config": config_dict(cfg, world),
                 "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle_threads(), "kind": "oracle",
                                  "sample": sample},
                 "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}})
    return base


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest value over the ranks (the slowest replica's time), through
    an all-reduce on the default process group; the value itself on one rank."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, units_per_rank: float, ms: float) -> float:
    """Units per second processed by all replicas together in ms milliseconds
    (weak scaling: every rank processes units_per_rank)."""
    return world * units_per_rank / (ms / 1e3)


def config_dict(cfg, world):
    return {"workload": f"{cfg.name}: T={cfg.T} H={cfg.H} I={cfg.I} E={cfg.E} top_k={cfg.k} block_size={cfg.bs} "
                        f"act={cfg.act} weights={cfg.wfmt}" + (f" lora_rank={cfg.lora_rank}" if cfg.lora_rank else ""),
            "T": cfg.T, "H": cfg.H, "I": cfg.I, "E": cfg.E, "top_k": cfg.k, "block_size": cfg.bs,
            "weights": cfg.wfmt, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": "inputs larger than L2 (all expert weights stream from HBM every step)"}


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

def run_ours(args, cfg, rank, world, local_rank):
    import numpy as np
    import torch
    import torch.distributed as dist

    from mixture_experts_grouped_gb300 import build as B
    from mixture_experts_grouped_gb300 import layer as L
    from mixture_experts_grouped_gb300 import moe as M
    from mixture_experts_grouped_gb300 import synth

    if not os.path.exists(M.LIB_PATH):
        B.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    inp = synth.make_inputs(cfg)
    wgu = L.upload_weight(inp["w_gate_up"], cfg.act, dev)
    wd = L.upload_weight(inp["w_down"], cfg.act, dev)
    dl = L.upload_lora(inp["lora"], cfg.I, cfg.H, dev) if inp["lora"] is not None else None
    lay = L.MoeLayer(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.bs, cfg.act, wgu, wd, dev, lora=dl,
                     renormalize=cfg.renormalize)
    x = L.act_tensor(inp["x"], cfg.act, dev)
    logits = torch.from_numpy(inp["logits"]).to(dev)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # the layer is captured once as CUDA graphs (it has no host synchronisation):
    # pre = route + align, gate_up, post = down + fold + combine
    g_pre, g_gu, g_post, g_all, per_step = lay.capture(x, logits)
    for _ in range(args.warmup):
        g_pre.replay()
        g_gu.replay()
        g_post.replay()
    torch.cuda.synchronize()
    if int(lay.err.item()) != 0:
        raise RuntimeError(f"device error word {int(lay.err.item()):#x} after warm-up")
    alg = algorithmic(cfg, lay.topk_ids.cpu().numpy())

    # ---- device-timed region: K steps, each one replay of the whole layer ----
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cvd = [c for c in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if c.strip()]
    phys = int(cvd[local_rank]) if local_rank < len(cvd) and cvd[local_rank].strip().isdigit() else local_rank
    clocks = ClockSampler(phys)
    barrier()
    clocks.start()
    time.sleep(0.3)  # let the sampler attach
    t_start.record(stream)
    for _ in range(args.steps):
        g_all.replay()
    t_end.record(stream)
    barrier()
    n_launch = per_step * args.steps
    ms = t_start.elapsed_time(t_end)
    # ---- kernel-timed region: K more steps as three graphs, events around gate/up ----
    ev_gu = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    s0.record(stream)
    for i in range(args.steps):
        g_pre.replay()
        ev_gu[i][0].record(stream)
        g_gu.replay()
        ev_gu[i][1].record(stream)
        g_post.replay()
    s1.record(stream)
    barrier()
    clk = clocks.stop()
    gu_ms = sum(a.elapsed_time(b) for a, b in ev_gu) / args.steps
    split_ms = s0.elapsed_time(s1) / args.steps
    ms = max_over_ranks(ms, world, dev)
    ms_per_step = ms / args.steps
    tokens_per_s = whole_job_rate(world, cfg.T * args.steps, ms)

    # ---- end to end through the public API: pinned host in, host out ----
    x_host = x.cpu().pin_memory()
    lg_host = logits.cpu().pin_memory()
    out_host = torch.empty(lay.out.shape, dtype=lay.out.dtype).pin_memory()
    x_dev = torch.empty_like(x)
    lg_dev = torch.empty_like(logits)
    n_e2e = max(3, min(args.steps, 200))
    for _ in range(3):
        x_dev.copy_(x_host, non_blocking=True)
        lg_dev.copy_(lg_host, non_blocking=True)
        lay.forward(x_dev, lg_dev)
        out_host.copy_(lay.out, non_blocking=True)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n_e2e):
        x_dev.copy_(x_host, non_blocking=True)
        lg_dev.copy_(lg_host, non_blocking=True)
        lay.forward(x_dev, lg_dev)
        out_host.copy_(lay.out, non_blocking=True)
    e1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    e2e_value = whole_job_rate(world, cfg.T * n_e2e, e2e_ms)
    if int(lay.err.item()) != 0:
        raise RuntimeError(f"device error word {int(lay.err.item()):#x}")
    if rank != 0:
        return None

    pk, pk_kind = peaks()
    peak_tf, peak_name = tensor_peak(pk, clk)
    tflops = alg["flops"] / (ms_per_step / 1e3) / 1e12
    weight_gbs = alg["weight_bytes"] / (ms_per_step / 1e3) / 1e9
    hbm = float(pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    layer_frac = max(tflops / peak_tf, (alg["bytes"] / (ms_per_step / 1e3) / 1e9) / hbm)
    # the dominant kernel's bound: tensor above the ridge point, HBM below it
    intensity = alg["flops_gate_up"] / alg["gate_up_bytes"]
    ridge = peak_tf * 1e12 / (hbm * 1e9)
    if intensity >= ridge:
        roof = {"bound": "tensor", "achieved": alg["flops_gate_up"] / (gu_ms / 1e3) / 1e12, "peak": peak_tf,
                "unit": "TFLOP/s", "peak_kind": f"bf16 dense {peak_name}, {pk_kind}"}
    else:
        roof = {"bound": "hbm", "achieved": alg["gate_up_bytes"] / (gu_ms / 1e3) / 1e9, "peak": hbm,
                "unit": "GB/s", "peak_kind": f"HBM copy, {pk_kind}"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    line = {
        "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": cfg.act, "data": "synthetic (seeded)",
        "config": config_dict(cfg, world),
        "tflops": tflops, "weight_gbs": weight_gbs, "layer_roofline_frac": layer_frac,
        "roofline": dict(roof, kernel="moe_grouped_gate_up (activation gather + tcgen05 grouped GEMM, fused "
                                       "SiLU-mul)",
                         traffic=traffic_for("grouped_gemm_gate_up", config_dict(cfg, world)["workload"]), ms_per_launch=gu_ms,
                         flops_per_launch=alg["flops_gate_up"], bytes_per_launch=alg["gate_up_bytes"],
                         intensity_flop_per_byte=intensity),
        "e2e": {"value": e2e_value, "unit": "tokens/s",
                "h2d_bytes_per_step": x_host.numel() * x_host.element_size() + lg_host.numel() * 4,
                "d2h_bytes_per_step": out_host.numel() * out_host.element_size(), "steps": n_e2e},
        "gpu_launches": int(n_launch),
        "launch_mode": f"CUDA graph of the whole layer, {per_step} kernels per step; roofline.ms_per_launch from a "
                       f"second timed region of {args.steps} steps replayed as three graphs with CUDA events "
                       f"around the gate/up call",
        "ms_per_step_three_graphs": split_ms,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, args.cpu_seconds, inp)
    return line


def run_fold(args, cfg):
    """The decode LoRA fold alone: moe_lora_gather_bgmv on the T * top_k
    slot-major rows of the workload (x = post-SiLU rows [P, I], base = down
    outputs [P, H]), expert ids from the library's own routing of the
    workload's logits. Reports algorithmic bytes per launch over the
    CUDA-event time against the HBM peak."""
    import numpy as np
    import torch

    from mixture_experts_grouped_gb300 import build as B
    from mixture_experts_grouped_gb300 import layer as L
    from mixture_experts_grouped_gb300 import moe as M
    from mixture_experts_grouped_gb300 import synth

    if not os.path.exists(M.LIB_PATH):
        B.build()
    assert cfg.lora_rank > 0, "--fold-only needs a workload with a LoRA rank"
    dev = torch.device("cuda", 0)
    inp = synth.make_inputs(cfg)
    lora = inp["lora"]
    dl = L.upload_lora(lora, cfg.I, cfg.H, dev)
    P = cfg.P
    logits = torch.from_numpy(inp["logits"]).to(dev)
    ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=dev)
    w = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=dev)
    M.moe_route_topk_softmax(logits, ids, w, cfg.T, cfg.E, cfg.k, cfg.renormalize)
    g = torch.Generator(device="cpu").manual_seed(0)
    x = torch.randn((P, cfg.I), generator=g).to(torch.bfloat16).to(dev)
    base = torch.randn((P, cfg.H), generator=g).to(torch.bfloat16).to(dev)
    xa = torch.zeros((P, dl.route.max_rank), dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize()
    e_host = ids.reshape(-1).cpu().numpy()
    adapted = np.array([e < lora["n_experts"] and e in lora["a"] for e in e_host])
    F = int(adapted.sum())
    U = len(set(e_host[adapted].tolist()))
    r = dl.route.max_rank
    bytes_per = (F * cfg.I * 2 + U * (r * cfg.I * 2 + cfg.H * r * 2) + F * r * 2 * 2 + F * cfg.H * 2 * 2 + P * 4)

    def launch():
        M.moe_lora_gather_bgmv(dl.route, x, base, ids, None, xa, P, cfg.k, 0)

    for _ in range(args.warmup):
        launch()
    torch.cuda.synchronize()
    # replayed from a CUDA graph of R folds, so that host launch cost is not timed
    R = 20
    reps = max(1, args.steps // R)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        launch()
    torch.cuda.current_stream().wait_stream(side)
    n_cap = M.moe_launch_count()
    with torch.cuda.graph(graph):
        for _ in range(R):
            launch()
    per_graph = M.moe_launch_count() - n_cap
    graph.replay()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(reps):
        graph.replay()
    e1.record(st)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (reps * R)
    launches = per_graph * reps
    pk, src = peaks()
    gbs = bytes_per / (ms * 1e-3) / 1e9
    return {
        "metric": "decode LoRA fold (moe_lora_gather_bgmv) algorithmic GB/s", "value": round(gbs, 2),
        "unit": "GB/s", "n_gpus": 1, "steps": reps * R, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{cfg.name}: n_slots={P} k_in={cfg.I} n_out={cfg.H} rank={r} "
                               f"folded_rows={F} adapted_experts_touched={U}",
                   "l2": "back-to-back folds from a CUDA graph; the fold's working set fits in L2"},
        "roofline": {"bound": "hbm", "achieved": round(gbs, 2), "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(gbs / pk["hbm_gbs"], 4), "peak_source": src, "bytes_per_launch": bytes_per},
        "gpu_launches": launches,
    }


# FP32 fused multiply-add peak of the CUDA cores: 152 SMs x 128 lanes x 2 FLOP
# x 2.07 GHz (maximum SM clock), the bound of the router GEMM
ALU_FP32_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def run_router(args, cfg):
    """The router GEMM and routing alone (moe_router_topk_softmax): logits =
    x . Wr with the workload's router weight (a router="gemm" workload), then
    the top-k softmax. Replayed from CUDA graphs of 20 calls."""
    import torch

    from mixture_experts_grouped_gb300 import build as B
    from mixture_experts_grouped_gb300 import layer as L
    from mixture_experts_grouped_gb300 import moe as M
    from mixture_experts_grouped_gb300 import synth

    if not os.path.exists(M.LIB_PATH):
        B.build()
    assert cfg.router == "gemm", "--router-only needs a workload with a router weight (router=gemm)"
    dev = torch.device("cuda", 0)
    a = synth.make_activations(cfg)
    x = L.act_tensor(a["x"], cfg.act, dev)
    wr = torch.from_numpy(a["w_router"]).to(dev)
    logits = torch.empty((cfg.T, cfg.E), dtype=torch.float32, device=dev)
    ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=dev)
    w = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=dev)

    def launch():
        M.moe_router_topk_softmax(x, M.ACT_CODES[cfg.act], wr, cfg.T, cfg.H, cfg.E, cfg.k, cfg.renormalize, logits,
                                  ids, w)

    for _ in range(args.warmup):
        launch()
    torch.cuda.synchronize()
    R = 20
    reps = max(1, args.steps // R)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        launch()
    torch.cuda.current_stream().wait_stream(side)
    n_cap = M.moe_launch_count()
    with torch.cuda.graph(graph):
        for _ in range(R):
            launch()
    per_graph = M.moe_launch_count() - n_cap
    graph.replay()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(reps):
        graph.replay()
    e1.record(st)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (reps * R)
    flops = 2.0 * cfg.T * cfg.H * cfg.E
    # bytes the call must move: x read once, the router weight, logits, ids and weights written
    nbytes = cfg.T * cfg.H * 2 + cfg.H * cfg.E * 4 + cfg.T * cfg.E * 4 + cfg.T * cfg.k * 8
    tf = flops / (ms * 1e-3) / 1e12
    gbs = nbytes / (ms * 1e-3) / 1e9
    pk, src = peaks()
    hbm = float(pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    # the bound: HBM below the fp32 ridge (ALU peak / HBM peak, about 12 FLOP/B), ALU above it
    if flops / nbytes < ALU_FP32_TFLOPS * 1e12 / (hbm * 1e9):
        roof = {"bound": "hbm", "achieved": round(gbs, 2), "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4),
                "peak_source": f"HBM copy, {src}", "bytes_per_call": nbytes}
    else:
        roof = {"bound": "alu", "achieved": round(tf, 3), "peak": round(ALU_FP32_TFLOPS, 1), "unit": "TFLOP/s",
                "frac": round(tf / ALU_FP32_TFLOPS, 4), "peak_source": "152 SMs x 128 FP32 lanes x 2 FLOP x 2.07 GHz",
                "flops_per_call": flops}
    return {
        "metric": "router GEMM + top-k softmax (moe_router_topk_softmax) us per call", "value": round(ms * 1e3, 3),
        "unit": "us", "n_gpus": 1, "steps": reps * R, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": False, "dtype": "f32 (bf16/fp16 activations)", "data": "synthetic",
        "config": {"workload": f"{cfg.name}: T={cfg.T} H={cfg.H} E={cfg.E} top_k={cfg.k} act={cfg.act}",
                   "l2": "back-to-back calls from a CUDA graph"},
        "tflops": round(tf, 3), "gbs": round(gbs, 2),
        "roofline": roof,
        "gpu_launches": per_graph * reps,
    }


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    cfg = workload(args.workload)
    if args.override:
        from dataclasses import replace
        kv = dict(item.split("=") for item in args.override.split(","))
        cfg = replace(cfg, name=f"{cfg.name}[{args.override}]",
                      **{k: type(getattr(cfg, k))(v) for k, v in kv.items()})
    if args.router_only:
        line = run_router(args, cfg) if rank == 0 else None
    elif args.fold_only:
        line = run_fold(args, cfg) if rank == 0 else None
    elif args.impl == "reference":
        line = run_reference(args, cfg, rank, world)
    else:
        if world > 1:
            import torch
            import torch.distributed as dist
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        line = run_ours(args, cfg, rank, world, local_rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
