"""Benchmark of the sparse top-k MoE training step on GB300.

One step = one full pass of the training step (router, dispatch, expert MLPs,
combine, MSE + aux losses, the full backward including dX, SGD) through the C
ABI entry point moe_train_step, on one synthetic batch already resident in HBM.

Prints ONE JSON line (rank 0).  Default workload: the large layer (T=65536,
D=4096, E=128, k=8, SwiGLU F=2048, bf16 with fp32 masters).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the float64 CPU oracle on a sample

N > 1 (under torchrun): every rank runs an independent replica of the step on
its own GPU (replicas only: the layer has no cross-GPU exchange step here);
value = all ranks' tokens / the slowest rank's time.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time
from typing import Optional

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "MoE train-step tokens/sec (fwd+bwd+SGD) at 1 GB300; expert-GEMM TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
GB300_SMS = 152
FFMA_PER_SM_PER_CLK = 128


# DRAM bytes of the expert GEMM family per training step of the large layer,
# from an ncu capture (dram__bytes_read.sum + dram__bytes_write.sum) of the
# same per-expert shapes at 8 experts, scaled by 16.  Valid only for the GEMM
# source it was taken from: reported as null once gemm_tc.cu changes.
GEMM_TRAFFIC = {"bytes_per_step": 107.4e9, "workload": "large",
                "gemm_source_sha256_prefix": "f575d8870daa70d5", "gradients_stored": False}


def gemm_traffic(wl: W.Workload, store_grads: bool = False):
    import hashlib
    src = os.path.join(ROOT, "sparse_mixture_experts_softmax_gb300", "csrc", "gemm_tc.cu")
    try:
        with open(src, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()
    except OSError:
        return None
    if wl.name != GEMM_TRAFFIC["workload"] or not sha.startswith(GEMM_TRAFFIC["gemm_source_sha256_prefix"]):
        return None
    if store_grads != GEMM_TRAFFIC["gradients_stored"]:
        return None
    return GEMM_TRAFFIC["bytes_per_step"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    d = dict(FALLBACK_PEAKS)
    d["source"] = "fallback"
    return d


def expert_flops_per_step(wl: W.Workload, rows: Optional[int] = None) -> float:
    """Algorithmic active-row FLOPs of the expert GEMMs in one training step:
    per routed row 2*D*F per projection, SwiGLU has 3 projections (W1, W3, W2),
    the two-layer MLP 2; backward is twice the forward.  ``rows``: the rows
    the experts process (fewer than T k when a capacity drops some)."""
    proj = 3 if wl.act == "swiglu" else 2
    return 3.0 * proj * 2.0 * wl.D * wl.F * (wl.R if rows is None else rows)


def gemm_launch_flops(wl: W.Workload, rows: Optional[int] = None) -> dict:
    """Algorithmic FLOPs per training step of each named expert-GEMM launch
    (2 flops per multiply-add over the rows the experts process).  The SwiGLU
    up-projection multiplies by W1 and W3 in one launch; the dX launch sums
    dH1 W1 + dH3 W3.  Summed, they give ``expert_flops_per_step``."""
    R = wl.R if rows is None else rows
    one = 2.0 * R * wl.D * wl.F
    if wl.act == "swiglu" and wl.dtype == "bf16":
        return {"gemm_up": 2 * one, "gemm_down": one, "gemm_dA": one, "gemm_dw2": one,
                "gemm_dxe": 2 * one, "gemm_dw1": one, "gemm_dw3": one}
    if wl.act == "swiglu":
        return {"gemm_up": one, "gemm_up_w3": one, "gemm_down": one, "gemm_dA": one,
                "gemm_dw2": one, "gemm_dxe": 2 * one, "gemm_dw1": one, "gemm_dw3": one}
    return {"gemm_up": one, "gemm_down": one, "gemm_dA": one, "gemm_dw2": one,
            "gemm_dxe": one, "gemm_dw1": one}


def shared_flops_per_step(wl: W.Workload) -> float:
    """The shared-expert branch (reported separately from the routed experts):
    three projections of 2*T*D*(n_shared*F) FLOPs, forward and twice that in
    backward."""
    return 3.0 * 3.0 * 2.0 * wl.T * wl.D * wl.n_shared * wl.F


def router_flops_per_step(wl: W.Workload) -> float:
    return 3.0 * 2.0 * wl.T * wl.D * wl.E


def hbm_bytes(wl: W.Workload, rows: Optional[int] = None) -> dict:
    """Algorithmic bytes per launch of the HBM-bound passes (``rows``: expert
    rows kept, T k without a capacity)."""
    es = 2 if wl.dtype == "bf16" else 4
    T, D, R = wl.T, wl.D, (wl.R if rows is None else rows)
    n_exp = (3 if wl.act == "swiglu" else 2) * wl.E * wl.D * wl.F
    n_bias = wl.E * (wl.F + wl.D) if wl.has_bias else 0
    return {
        "gather": T * D * es + R * D * es,                 # X once, Xe written
        "combine_loss": R * D * es + 2 * T * D * 4,       # Ye, target read; dY written
        "combine_bwd": T * D * 4 + 2 * R * D * es,        # dY, Ye read; dYe written
        # training step (k <= 8): combine, MSE seed and combine backward in one
        # pass: Ye and the target read, dYe written
        "combine_fused": 2 * R * D * es + T * D * 4,
        # dX = router term + sum_j dXe[slot(t, j)]: dXe read, dX read and written
        "scatter_back": R * D * es + 2 * T * D * 4,
        # the stand-alone SGD launches: master and gradient read, master
        # written.  bf16 layers update the expert weights inside the dW GEMM
        # epilogues, so only the router weight and biases remain here.
        "sgd": (wl.E * D + n_bias + (0 if wl.dtype == "bf16" else n_exp)) * 12,
    }


def max_over_ranks(x: float, device) -> float:
    """The largest of every rank's x (x itself with a single process)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, world: int, steps: int, seconds: float) -> float:
    """Units all ranks processed over the slowest rank's time (weak scaling:
    every rank runs its own replica of the step on its own batch)."""
    return units_per_rank * world * steps / seconds


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
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
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def oracle_sample_step(wl: W.Workload, T_s: int, E_s: int, seed: int = 0):
    """One oracle training step on a bounded sample of the workload: T_s tokens
    of the same layer width (D, F, k, activation, scores) over its first E_s
    experts.  Returns (seconds, description)."""
    import numpy as np
    import torch
    from oracle import moe_oracle as O

    E_s = max(E_s, wl.k)
    if wl.n_groups > 1:
        per = wl.E // wl.n_groups
        E_s = max(E_s, per * wl.topk_groups)
        E_s = (E_s + per - 1) // per * per
    n_groups = wl.n_groups if wl.n_groups == 1 else E_s // (wl.E // wl.n_groups)
    topk_groups = min(wl.topk_groups, n_groups)
    sub = W.Workload(wl.name + "_sample", T=T_s, D=wl.D, F=wl.F, E=E_s, k=wl.k, act=wl.act,
                     score=wl.score, n_groups=n_groups, topk_groups=topk_groups,
                     has_bias=wl.has_bias, dtype=wl.dtype, aux_alpha=wl.aux_alpha, lr=wl.lr,
                     router_init=wl.router_init, corr_bias_scale=wl.corr_bias_scale,
                     n_shared=wl.n_shared, capacity_factor=wl.capacity_factor)
    inp = W.make_inputs(sub, seed=seed)
    f64 = lambda t: None if t is None else t.detach().double().numpy()  # noqa: E731
    lp = wl.dtype == "bf16"
    w = dict(w_gate=f64(inp["w_gate"].to(torch.bfloat16) if lp else inp["w_gate"]),
             w1=f64(inp["w1_bf16"] if lp else inp["w1"]),
             w2=f64(inp["w2_bf16"] if lp else inp["w2"]),
             w3=f64(inp["w3_bf16"] if lp and inp["w3"] is not None else inp["w3"]),
             b1=f64(inp["b1"]), b2=f64(inp["b2"]), logit_bias=None,
             corr_bias=f64(inp.get("corr_bias")))
    if wl.n_shared > 0:
        for key in ("ws1", "ws3", "ws2"):
            w[key] = f64(inp[key + "_bf16"] if lp else inp[key])
    x = f64(inp["x_bf16"] if lp else inp["x"])
    tgt = f64(inp["target"])
    cfg = O.OracleConfig(T=T_s, D=wl.D, F=wl.F, E=E_s, k=wl.k, act=wl.act, score=wl.score,
                         n_groups=n_groups, topk_groups=topk_groups, has_bias=wl.has_bias,
                         aux_alpha=wl.aux_alpha, capacity_factor=wl.capacity_factor)
    # the oracle's train step, its SGD timed apart: the same calls as
    # O.train_step, in its order
    t0 = time.perf_counter()
    st = O.forward(cfg, w, x)
    _, _, dy = O.losses(cfg, st, tgt)
    grads = O.backward(cfg, w, x, st, dy)
    t1 = time.perf_counter()
    O.sgd(w, grads, wl.lr)
    t2 = time.perf_counter()
    desc = (f"oracle train step (fwd+bwd+SGD, float64 numpy) on {T_s} tokens of the "
            f"{wl.name} layer (D={wl.D}, F={wl.F}, k={wl.k}) over {E_s} of its {wl.E} experts")
    return t1 - t0, t2 - t1, desc


def extrapolated_rate(wl: W.Workload, T_s: int, E_s: int, t_tok: float, t_sgd: float) -> float:
    """Tokens/s of a whole step of the workload from a sample: the per-token
    part (router, dispatch, experts, combine, losses, backward) scales with T
    / T_s; the SGD part updates every parameter once per step and scales with
    the E / E_s experts (router and biases included in that share)."""
    return wl.T / (t_tok * wl.T / T_s + t_sgd * wl.E / E_s)


def sample_size(wl: W.Workload):
    """Tokens / experts of the CPU sample: about 10-30 s of float64 work."""
    per_tok = 3 * (3 if wl.act == "swiglu" else 2) * 2 * wl.D * wl.F * wl.k
    per_tok += 3 * 3 * 2 * wl.D * wl.n_shared * wl.F      # shared-expert branch
    T_s = int(max(16, min(wl.T, 2.0e11 / per_tok)))
    E_s = min(wl.E, 16)
    return T_s, E_s


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, wl):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    T_s, E_s = sample_size(wl)
    tok, sgd = [], []
    desc = ""
    for i in range(args.warmup + args.steps):
        t_tok, t_sgd, desc = oracle_sample_step(wl, T_s, E_s)
        if i >= args.warmup:
            tok.append(t_tok)
            sgd.append(t_sgd)
    t_tok, t_sgd = sum(tok) / len(tok), sum(sgd) / len(sgd)
    value = extrapolated_rate(wl, T_s, E_s, t_tok, t_sgd)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * wl.T / value, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(),
                             "kind": "oracle", "sample": desc,
                             "extrapolated": extrapolation_note(wl, T_s, E_s, t_tok, t_sgd)},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def extrapolation_note(wl, T_s, E_s, t_tok, t_sgd) -> str:
    return (f"extrapolated from a sample: whole-step time = {t_tok:.3f} s x {wl.T}/{T_s} tokens "
            f"+ SGD {t_sgd:.3f} s x {wl.E}/{E_s} experts")


def workload_config(wl: W.Workload) -> dict:
    return {"workload": wl.name, "tokens": wl.T, "d_model": wl.D, "d_ff": wl.F, "experts": wl.E,
            "top_k": wl.k, "activation": wl.act, "scores": wl.score, "n_groups": wl.n_groups,
            "topk_groups": wl.topk_groups, "expert_dtype": wl.dtype, "aux_alpha": wl.aux_alpha,
            "lr": wl.lr, "global_batch": wl.T, "parallelism": "replicas",
            "n_shared": wl.n_shared, "corr_bias": wl.corr_bias_scale is not None,
            "capacity_factor": wl.capacity_factor,
            "l2": "inputs larger than L2 (weights and expert-major activations >> 129 MB)"}


def routing_summary(layer, wl: W.Workload) -> dict:
    """Realised load of the step's routing: the share of the T k assignments
    taken by the three busiest experts, the largest and smallest expert
    loads, and the experts that received none."""
    counts = sorted((int(c) for c in layer.routing()["counts"].cpu().tolist()), reverse=True)
    R = max(wl.T * wl.k, 1)
    return {"top3_share": round(sum(counts[:3]) / R, 4), "max_rows": counts[0],
            "min_rows": counts[-1], "empty_experts": sum(1 for c in counts if c == 0)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="large", choices=sorted(W.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--kernels", action="store_true", help="print per-kernel times to stderr")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override T (profiling a smaller case of the same layer)")
    ap.add_argument("--experts", type=int, default=None,
                    help="override E (profiling a smaller case of the same layer)")
    ap.add_argument("--store-grads", action="store_true",
                    help="hand out every fp32 gradient (default: the step applies them "
                         "in the fused SGD without storing them)")
    args = ap.parse_args()
    wl = W.WORKLOADS[args.workload]
    if args.tokens is not None or args.experts is not None:
        import dataclasses
        wl = dataclasses.replace(wl, T=args.tokens or wl.T, E=args.experts or wl.E,
                                 zipf_empty=min(wl.zipf_empty, max(0, (args.experts or wl.E) - wl.k)),
                                 name=f"{wl.name}(T={args.tokens or wl.T},E={args.experts or wl.E})")
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args, wl)
        return

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    from sparse_mixture_experts_softmax_gb300 import binding as B
    from sparse_mixture_experts_softmax_gb300.layer import MoELayer

    inp = W.make_inputs(wl, seed=rank, device=str(dev))   # each replica its own batch
    lp = wl.dtype == "bf16"
    layer = MoELayer(wl.T, wl.D, wl.F, wl.E, wl.k, wl.act, wl.score, wl.dtype, wl.has_bias,
                     wl.aux_alpha, inp["w_gate"], inp["w1"], inp["w2"], w3=inp["w3"],
                     b1=inp["b1"], b2=inp["b2"], logit_bias=inp["logit_bias"],
                     n_groups=wl.n_groups, topk_groups=wl.topk_groups,
                     w1_lp=inp.get("w1_bf16"), w3_lp=inp.get("w3_bf16"),
                     w2_lp=inp.get("w2_bf16"), device=str(dev), corr_bias=inp.get("corr_bias"),
                     n_shared=wl.n_shared, ws1=inp.get("ws1"), ws3=inp.get("ws3"),
                     ws2=inp.get("ws2"), capacity_factor=wl.capacity_factor,
                     store_grads=args.store_grads)
    x = (inp["x_bf16"] if lp else inp["x"]).contiguous()
    tgt = inp["target"].contiguous()
    dx = torch.empty(wl.T, wl.D, device=dev)
    for k_ in ("w1", "w2", "w3", "w1_bf16", "w2_bf16", "w3_bf16", "ws1", "ws3", "ws2",
               "ws1_bf16", "ws3_bf16", "ws2_bf16"):
        inp.pop(k_, None)
    torch.cuda.empty_cache()

    # warm-up steps, each timed on its own (the first one includes the
    # one-time costs: module load, tensor-map encoding, attribute setup)
    warm_ms = []
    for _ in range(args.warmup):
        a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_ev.record()
        layer.train_step(x, tgt, wl.lr, dx=dx)
        b_ev.record()
        torch.cuda.synchronize()
        warm_ms.append(a_ev.elapsed_time(b_ev))
    launches = B.moe_last_launch_count()

    stream = torch.cuda.current_stream()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    # the timed region: K steps with nothing recorded between their launches
    # but one event per step boundary
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps - 1)]
    start.record(stream)
    for i in range(args.steps):
        layer.train_step(x, tgt, wl.lr, dx=dx)
        if i < args.steps - 1:
            step_ev[i].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    marks = [start] + step_ev + [end]
    step_ms = sorted(marks[i].elapsed_time(marks[i + 1]) for i in range(args.steps))
    if world > 1:
        dist.barrier()
    ms_total = start.elapsed_time(end)
    # the per-kernel breakdown: K more steps with a CUDA event pair around
    # every launch (the events cost a little time between launches, so these
    # steps are not the timed ones)
    B.moe_profile_enable(True)
    for i in range(args.steps):
        layer.train_step(x, tgt, wl.lr, dx=dx)
    torch.cuda.synchronize()
    clk = clocks.stop()
    prof = B.moe_profile_read()
    B.moe_profile_enable(False)
    ms_total = max_over_ranks(ms_total, dev)
    ms_step = ms_total / args.steps
    value = whole_job_rate(wl.T, world, args.steps, ms_total / 1e3)
    loss = layer.d_loss.cpu().tolist()

    # per-kernel times over the profiled steps
    per_kernel = {}
    for name, ms in prof:
        per_kernel[name] = per_kernel.get(name, 0.0) + ms
    for k_ in per_kernel:
        per_kernel[k_] /= args.steps
    gemm_ms = sum(v for k_, v in per_kernel.items()
                  if k_.startswith("gemm_") and not k_.startswith(("gemm_router", "gemm_shared")))
    shared_ms = sum(v for k_, v in per_kernel.items() if k_.startswith("gemm_shared"))
    peaks = load_peaks()
    rows_kept = int(layer.routing()["offsets"][-1].item())   # T k unless a capacity drops
    eflops = expert_flops_per_step(wl, rows_kept)
    # fp32 layers on the tensor cores do six bf16 term products per fp32
    # product (csrc/gemm_f32x3.cu): their roofline counts that tensor work
    path = B.moe_expert_gemm_path(layer.cfg)
    f32x3 = (not lp) and path == B.GEMM_TENSOR_F32X3
    work = 6.0 if f32x3 else 1.0
    mhz = clk.get("sm_max_mhz") or 2070.0
    ffma_peak = GB300_SMS * FFMA_PER_SM_PER_CLK * 2 * mhz * 1e6 / 1e12
    if lp or f32x3:
        achieved = work * eflops / (gemm_ms / 1e3) / 1e12
        peak = float(peaks["bf16_tflops_sustained"])
        bound, unit = "tensor", "TFLOP/s"
    else:
        achieved = eflops / (gemm_ms / 1e3) / 1e12
        peak = ffma_peak
        bound, unit = "alu", "TFLOP/s"
    roofline = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak, "traffic": gemm_traffic(wl, args.store_grads),
                "traffic_unit": "DRAM bytes per step of the GEMM family",
                "traffic_measured_in_this_run": False,
                "traffic_source": ("ncu dram__bytes_read.sum + dram__bytes_write.sum of every "
                                   "expert-GEMM launch at 8 experts, scaled by 16 "
                                   "(profiles/tc_gemm_large_e8_traffic.md); null when the GEMM "
                                   "source differs from the one captured"),
                "kernel": "grouped expert GEMMs (all launches of one step)",
                "peak_source": f"{peaks['source']} "
                               f"({'bf16_tflops_sustained' if (lp or f32x3) else 'FFMA at max clock'})"}
    if lp or f32x3:
        burst = float(peaks["bf16_tflops"])
        roofline["peak_burst"] = burst
        roofline["frac_of_burst"] = achieved / burst
    if f32x3:
        eff = eflops / (gemm_ms / 1e3) / 1e12
        roofline["kernel"] = ("grouped expert GEMMs of an fp32 layer on the tensor cores: each fp32 "
                              "operand split into three bf16 terms, six term products per fp32 "
                              "product (counted in `achieved`), operand expansion and activation "
                              "passes included in the time")
        roofline["fp32_effective_tflops"] = eff
        roofline["fp32_effective_vs_ffma_peak"] = eff / ffma_peak
    roofline["gemm_path"] = {B.GEMM_CUDA_CORES: "cuda_cores", B.GEMM_TENSOR_BF16: "tensor_bf16",
                             B.GEMM_TENSOR_F32X3: "tensor_fp32_three_term_split"}.get(path, "?")
    # each expert-GEMM launch on its own (FLOPs per step / its time per step)
    launches_tc = {}
    for name, fl in gemm_launch_flops(wl, rows_kept).items():
        ms = per_kernel.get(name, 0.0)
        if ms > 0:
            tf = work * fl / (ms / 1e3) / 1e12
            launches_tc[name] = {"ms": round(ms, 4), "TFLOP/s": round(tf, 1),
                                 "frac": round(tf / peak, 4)}
            if lp or f32x3:
                launches_tc[name]["frac_of_burst"] = round(tf / float(peaks["bf16_tflops"]), 4)
    hb = hbm_bytes(wl, rows_kept)
    hbm = {}
    for name, key in (("gather", "gather"), ("combine_loss", "combine_loss"),
                      ("combine_bwd", "combine_bwd"), ("combine_fused", "combine_fused"),
                      ("scatter_back", "scatter_back")) + \
            ((("sgd", "sgd"),) if not lp else ()):
        if name in per_kernel and per_kernel[name] > 0:
            gbs = hb[key] / (per_kernel[name] / 1e3) / 1e9
            hbm[name] = {"ms": per_kernel[name], "GB/s": gbs, "frac": gbs / float(peaks["hbm_gbs"])}

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if lp else "f32", "data": "synthetic", "config": workload_config(wl),
            "expert_gemm_tflops": achieved, "router_gflop_per_step": router_flops_per_step(wl) / 1e9,
            "expert_gflop_per_step": eflops / 1e9, "expert_rows_per_step": rows_kept,
            "roofline": roofline, "gemm_launches": launches_tc, "hbm_passes": hbm,
            "routing": routing_summary(layer, wl),
            "gpu_launches": launches * args.steps, "clocks": clk,
            "step_ms": {"p50": step_ms[len(step_ms) // 2],
                        "p90": step_ms[min(len(step_ms) - 1, int(0.9 * len(step_ms)))],
                        "min": step_ms[0], "max": step_ms[-1]},
            "warmup_ms": [round(v, 3) for v in warm_ms],
            "loss": {"mse": loss[0], "aux": loss[1]},
            "kernels_ms_per_step": {k_: round(v, 4) for k_, v in sorted(per_kernel.items())}}
    line["config"]["gradients"] = (
        "every fp32 gradient stored" if args.store_grads else
        "applied by SGD, not handed out (NULL gradient buffers): bf16 layers update the "
        "expert weights inside the weight-gradient GEMMs and store no fp32 gradient")
    if wl.n_shared > 0 and shared_ms > 0:
        sf = shared_flops_per_step(wl)
        line["shared_experts"] = {"n_shared": wl.n_shared, "gflop_per_step": sf / 1e9,
                                  "ms_per_step": shared_ms, "tflops": sf / (shared_ms / 1e3) / 1e12}

    # end to end through the host-buffer entry point: every step uploads its
    # batch from pinned host memory and reads its losses back; the pipelined
    # call overlaps the upload of step i+1 with step i
    if not args.no_e2e:
        staging = torch.empty(2 * B.moe_host_staging_size(layer.cfg), dtype=torch.uint8,
                              device=dev)
        x_host = x.cpu().pin_memory()
        t_host = tgt.cpu().pin_memory()
        l_host = torch.zeros(2 * args.steps, dtype=torch.float32).pin_memory()
        B.moe_train_steps_host(layer.cfg, layer.params(), [x_host], [t_host], wl.lr, l_host,
                               staging, layer.workspace)   # warm-up (one step)
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        B.moe_train_steps_host(layer.cfg, layer.params(), [x_host] * args.steps,
                               [t_host] * args.steps, wl.lr, l_host, staging, layer.workspace)
        e2e_s = time.perf_counter() - t0
        e2e_s = max_over_ranks(e2e_s, dev)
        line["e2e"] = {"value": whole_job_rate(wl.T, world, args.steps, e2e_s), "unit": "tokens/s",
                       "h2d_bytes_per_step": x_host.numel() * x_host.element_size()
                       + t_host.numel() * 4, "d2h_bytes_per_step": 8,
                       "api": "moe_train_steps_host (upload of step i+1 overlapped with step i)"}

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        T_s, E_s = sample_size(wl)
        t_tok, t_sgd, desc = oracle_sample_step(wl, T_s, E_s)
        line["cpu_baseline"] = {"value": extrapolated_rate(wl, T_s, E_s, t_tok, t_sgd),
                                "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                                "sample": desc,
                                "extrapolated": extrapolation_note(wl, T_s, E_s, t_tok, t_sgd)}
    if args.kernels and rank == 0:
        for k_, v in sorted(per_kernel.items(), key=lambda kv: -kv[1]):
            print(f"{k_:20s} {v:9.3f} ms", file=sys.stderr)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
