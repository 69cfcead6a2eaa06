"""Seeded synthetic workloads for the sparse top-k MoE training step.

This module is shared by the float64 oracle (``oracle/``), the CUDA binding's
tests and ``bench.py``.  It holds only shapes, distributions and random draws:
none of the method's arithmetic (no routing, no expert math, no losses) lives
here, so neither side of a parity comparison can borrow the other's steps
through it.

Workloads follow the five configurations the layer is measured on (the course
"Trainable MoE in CUDA" names the method; the shapes and distributions are the
measurement configurations):

* ``tiny``        T=64,    D=32,   E=4,   k=2, F=64,   ReLU + biases, softmax, fp32, 20-step loop
* ``dense_f32``   T=4096,  D=512,  E=8,   k=2, F=1024, GELU(tanh) + biases, softmax, fp32
* ``dense_bf16``  the same layer with bf16 multiplicands
* ``grouped``     T=16384, D=1024, E=64 in 8 groups, top-4 groups, k=6, SwiGLU F=704,
                  sigmoid scores, no bias, bf16
* ``skewed``      T=32768, D=2048, E=64, k=8, SwiGLU F=1408, softmax with a fixed Zipf(1.2)
                  logit bias (4 experts never selected), bf16
* ``large``       T=65536, D=4096, E=128, k=8, SwiGLU F=2048, softmax, router U(+-1/sqrt(D)),
                  bf16 with fp32 master weights

Draw order (one ``torch.Generator`` seeded with ``seed``): W_g, W1, W3, W2,
A_teacher, X, eps; biases start at zero and are not drawn.  The Zipf rank
permutation of ``skewed`` comes from a second generator seeded ``seed + 1``.
``N(0, v)`` means variance ``v``: weights have std ``1/sqrt(fan_in)``, the target
noise std ``0.1``.  Targets are ``X @ A_teacher + eps`` with ``A_teacher ~
N(0, 1/D)``.  bf16 copies are round-to-nearest-even casts of the fp32 draws.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    D: int
    F: int
    E: int
    k: int
    act: str            # "relu" | "gelu_tanh" | "swiglu"
    score: str          # "softmax" | "sigmoid"
    n_groups: int
    topk_groups: int
    has_bias: bool
    dtype: str          # "f32" | "bf16"  (multiplicand type of the expert GEMMs)
    aux_alpha: float
    lr: float
    steps: int = 1
    router_init: str = "normal"      # "normal" -> N(0,1/D); "uniform" -> U(-1/sqrt(D), 1/sqrt(D))
    zipf_skew: Optional[float] = None  # Zipf exponent of the fixed logit bias
    zipf_empty: int = 0                # experts that get a -inf logit bias (never selected)
    corr_bias_scale: Optional[float] = None  # selection-only correction bias ~ U(-s, s)
    n_shared: int = 0                  # shared-expert SwiGLU branch of width n_shared * F
    capacity_factor: float = 0.0       # expert capacity ceil(cf T k / E); 0 = none

    @property
    def R(self) -> int:
        return self.T * self.k

    def with_tokens(self, T: int) -> "Workload":
        """The same layer on a different number of tokens (for sampled parity cases)."""
        return dataclasses.replace(self, T=T)


WORKLOADS = {
    "tiny": Workload("tiny", T=64, D=32, F=64, E=4, k=2, act="relu", score="softmax",
                     n_groups=1, topk_groups=1, has_bias=True, dtype="f32",
                     aux_alpha=0.01, lr=0.05, steps=20),
    "dense_f32": Workload("dense_f32", T=4096, D=512, F=1024, E=8, k=2, act="gelu_tanh",
                          score="softmax", n_groups=1, topk_groups=1, has_bias=True,
                          dtype="f32", aux_alpha=0.01, lr=0.01),
    "dense_bf16": Workload("dense_bf16", T=4096, D=512, F=1024, E=8, k=2, act="gelu_tanh",
                           score="softmax", n_groups=1, topk_groups=1, has_bias=True,
                           dtype="bf16", aux_alpha=0.01, lr=0.01),
    "grouped": Workload("grouped", T=16384, D=1024, F=704, E=64, k=6, act="swiglu",
                        score="sigmoid", n_groups=8, topk_groups=4, has_bias=False,
                        dtype="bf16", aux_alpha=0.0, lr=1e-3),
    "skewed": Workload("skewed", T=32768, D=2048, F=1408, E=64, k=8, act="swiglu",
                       score="softmax", n_groups=1, topk_groups=1, has_bias=False,
                       dtype="bf16", aux_alpha=0.01, lr=1e-3, zipf_skew=1.2, zipf_empty=4),
    "large": Workload("large", T=65536, D=4096, F=2048, E=128, k=8, act="swiglu",
                      score="softmax", n_groups=1, topk_groups=1, has_bias=False,
                      dtype="bf16", aux_alpha=0.01, lr=1e-3, router_init="uniform"),
    # correction-bias routing (selection on score + bias, gates from the scores)
    "grouped_cb": Workload("grouped_cb", T=16384, D=1024, F=704, E=64, k=6, act="swiglu",
                           score="sigmoid", n_groups=8, topk_groups=4, has_bias=False,
                           dtype="bf16", aux_alpha=0.0, lr=1e-3, corr_bias_scale=0.1),
    # shared experts (one SwiGLU branch of width n_shared * F on every token)
    "grouped_shared": Workload("grouped_shared", T=16384, D=1024, F=704, E=64, k=6,
                               act="swiglu", score="sigmoid", n_groups=8, topk_groups=4,
                               has_bias=False, dtype="bf16", aux_alpha=0.0, lr=1e-3, n_shared=2),
    "large_shared": Workload("large_shared", T=65536, D=4096, F=2048, E=128, k=8, act="swiglu",
                             score="softmax", n_groups=1, topk_groups=1, has_bias=False,
                             dtype="bf16", aux_alpha=0.01, lr=1e-3, router_init="uniform",
                             n_shared=1),
    # expert capacity (token dropping); factors exact in float32
    "skewed_cap": Workload("skewed_cap", T=32768, D=2048, F=1408, E=64, k=8, act="swiglu",
                           score="softmax", n_groups=1, topk_groups=1, has_bias=False,
                           dtype="bf16", aux_alpha=0.01, lr=1e-3, zipf_skew=1.2, zipf_empty=4,
                           capacity_factor=1.25),
    "dense_f32_cap": Workload("dense_f32_cap", T=4096, D=512, F=1024, E=8, k=2,
                              act="gelu_tanh", score="softmax", n_groups=1, topk_groups=1,
                              has_bias=True, dtype="f32", aux_alpha=0.01, lr=0.01,
                              capacity_factor=0.75),
    "dense_f32_cb": Workload("dense_f32_cb", T=4096, D=512, F=1024, E=8, k=2, act="gelu_tanh",
                             score="softmax", n_groups=1, topk_groups=1, has_bias=True,
                             dtype="f32", aux_alpha=0.01, lr=0.01, corr_bias_scale=0.05),
}


def _normal(shape, std, gen, device):
    return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32) * std


def zipf_logit_bias(wl: Workload, seed: int = 0) -> Optional[torch.Tensor]:
    """Fixed, non-trainable logit bias ``log(r^-s)`` over expert rank ``r``.

    Ranks ``1..E-zipf_empty`` go to expert ids through a seeded permutation (so
    the empty experts sit in the middle of the id range); the remaining
    ``zipf_empty`` experts get ``-inf`` and are never selected.  The constant
    ``-log(H)`` of the Zipf normaliser is dropped: it shifts every logit alike.
    """
    if wl.zipf_skew is None:
        return None
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 1)
    perm = torch.randperm(wl.E, generator=g)
    bias = torch.empty(wl.E, dtype=torch.float32)
    n_live = wl.E - wl.zipf_empty
    for rank0 in range(wl.E):
        e = int(perm[rank0])
        if rank0 < n_live:
            bias[e] = -wl.zipf_skew * math.log(rank0 + 1)
        else:
            bias[e] = float("-inf")
    return bias


def correction_bias(wl: Workload, seed: int = 0) -> Optional[torch.Tensor]:
    """Per-expert selection-only routing bias ~ U(-s, s), from its own seeded
    generator (so the other draws do not move), or None."""
    if wl.corr_bias_scale is None:
        return None
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 2)
    return (torch.rand(wl.E, generator=g) * 2.0 - 1.0) * wl.corr_bias_scale


def shared_weights(wl: Workload, seed: int = 0, device: str = "cpu") -> dict:
    """Shared-expert weights ws1, ws3 [n_shared F, D] ~ N(0, 1/D) and ws2
    [D, n_shared F] ~ N(0, 1/(n_shared F)) from their own seeded generator (so
    the other draws do not move), with bf16 copies for bf16 workloads; all
    None without shared experts."""
    keys = ("ws1", "ws3", "ws2", "ws1_bf16", "ws3_bf16", "ws2_bf16")
    if wl.n_shared <= 0:
        return {k_: None for k_ in keys}
    g = torch.Generator(device=device)
    g.manual_seed(seed + 3)
    Fs = wl.n_shared * wl.F
    ws1 = _normal((Fs, wl.D), 1.0 / math.sqrt(wl.D), g, device)
    ws3 = _normal((Fs, wl.D), 1.0 / math.sqrt(wl.D), g, device)
    ws2 = _normal((wl.D, Fs), 1.0 / math.sqrt(Fs), g, device)
    out = dict(ws1=ws1, ws3=ws3, ws2=ws2)
    lp = wl.dtype == "bf16"
    for k_ in ("ws1", "ws3", "ws2"):
        out[k_ + "_bf16"] = out[k_].to(torch.bfloat16) if lp else None
    return out


def make_inputs(wl: Workload, seed: int = 0, device: str = "cpu",
                with_target: bool = True) -> dict:
    """Draw one seeded workload.  Returns fp32 tensors plus bf16 copies.

    Keys: ``w_gate [E,D]``, ``w1 [E,F,D]``, ``w3 [E,F,D]`` (SwiGLU only, else
    None), ``w2 [E,D,F]``, ``b1 [E,F]`` / ``b2 [E,D]`` (zeros, or None without
    bias), ``logit_bias [E]`` or None, ``corr_bias [E]`` or None, ``x [T,D]`` fp32
    draws, ``target [T,D]``.
    For bf16 workloads ``x_bf16``, ``w1_bf16``, ``w3_bf16``, ``w2_bf16`` are the
    round-to-nearest-even casts; the fp32 expert weights are the master copy.
    """
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    T, D, F, E = wl.T, wl.D, wl.F, wl.E
    if wl.router_init == "uniform":
        a = 1.0 / math.sqrt(D)
        w_gate = (torch.rand(E, D, generator=g, device=device) * 2.0 - 1.0) * a
    else:
        w_gate = _normal((E, D), 1.0 / math.sqrt(D), g, device)
    w1 = _normal((E, F, D), 1.0 / math.sqrt(D), g, device)
    w3 = _normal((E, F, D), 1.0 / math.sqrt(D), g, device) if wl.act == "swiglu" else None
    w2 = _normal((E, D, F), 1.0 / math.sqrt(F), g, device)
    out = dict(w_gate=w_gate, w1=w1, w3=w3, w2=w2)
    out["b1"] = torch.zeros(E, F, device=device) if wl.has_bias else None
    out["b2"] = torch.zeros(E, D, device=device) if wl.has_bias else None
    a_teacher = _normal((D, D), 1.0 / math.sqrt(D), g, device)
    x = torch.randn(T, D, generator=g, device=device, dtype=torch.float32)
    out["x"] = x
    if with_target:
        eps = _normal((T, D), 0.1, g, device)
        out["target"] = x @ a_teacher + eps
    lb = zipf_logit_bias(wl, seed)
    out["logit_bias"] = lb.to(device) if lb is not None else None
    cb = correction_bias(wl, seed)
    out["corr_bias"] = cb.to(device) if cb is not None else None
    out.update(shared_weights(wl, seed, device))
    if wl.dtype == "bf16":
        out["x_bf16"] = x.to(torch.bfloat16)
        out["w1_bf16"] = w1.to(torch.bfloat16)
        out["w3_bf16"] = w3.to(torch.bfloat16) if w3 is not None else None
        out["w2_bf16"] = w2.to(torch.bfloat16)
    return out


def sample_tokens(T: int, n: int, seed: int = 0) -> torch.Tensor:
    """A seeded, sorted sample of ``n`` distinct token ids out of ``T``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 7)
    n = min(n, T)
    return torch.sort(torch.randperm(T, generator=g)[:n]).values
