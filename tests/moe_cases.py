"""Shared helpers of the parity tests: build the oracle's view and the CUDA
layer's view of one seeded workload, and compare them.

The oracle side receives exactly the values the CUDA side computes with:
fp32 draws for fp32 layers; for bf16 layers the bf16-rounded x and expert
weights (widened to float64), the bf16 copy of the router weight that the
router GEMM multiplies with, and the fp32 masters for the SGD update.  Nothing
the oracle consumes comes out of the CUDA library, except two kinds of
decision that floating point takes and that both sides must take in the
kernel's precision, each first validated against the oracle's own: a routing
(``validated_routing``: near-ties of the selection keys) and ReLU derivatives
at pre-activations within rounding of zero (``validated_relu_decisions``).
"""

from __future__ import annotations

import numpy as np
import torch

import workloads as W
from oracle import moe_oracle as O

TOL = {"f32": 1e-4, "bf16": 2e-2}


def oracle_config(wl: W.Workload, group_score="top2_sum") -> O.OracleConfig:
    return O.OracleConfig(T=wl.T, D=wl.D, F=wl.F, E=wl.E, k=wl.k, act=wl.act, score=wl.score,
                          n_groups=wl.n_groups, topk_groups=wl.topk_groups,
                          group_score=group_score, has_bias=wl.has_bias,
                          aux_alpha=wl.aux_alpha, capacity_factor=wl.capacity_factor)


def np64(t):
    if t is None:
        return None
    return t.detach().float().cpu().numpy().astype(np.float64)


def oracle_inputs(wl: W.Workload, inp: dict):
    """(weights used by forward/backward, fp32 master weights, x, target) in float64."""
    lp = wl.dtype == "bf16"
    # bf16 layers feed the router GEMM a bf16 copy of the fp32 master W_g
    w_fwd = dict(w_gate=np64(inp["w_gate"].to(torch.bfloat16) if lp else inp["w_gate"]),
                 w1=np64(inp["w1_bf16"] if lp else inp["w1"]),
                 w2=np64(inp["w2_bf16"] if lp else inp["w2"]),
                 w3=np64(inp["w3_bf16"] if lp else inp["w3"]) if inp["w3"] is not None else None,
                 b1=np64(inp["b1"]), b2=np64(inp["b2"]), logit_bias=np64(inp["logit_bias"]),
                 corr_bias=np64(inp.get("corr_bias")))
    master = dict(w_gate=np64(inp["w_gate"]), w1=np64(inp["w1"]), w2=np64(inp["w2"]),
                  w3=np64(inp["w3"]), b1=np64(inp["b1"]), b2=np64(inp["b2"]))
    if inp.get("ws1") is not None:   # shared-expert branch
        for key in ("ws1", "ws3", "ws2"):
            w_fwd[key] = np64(inp[key + "_bf16"] if lp else inp[key])
            master[key] = np64(inp[key])
    x = np64(inp["x_bf16"] if lp else inp["x"])
    return w_fwd, master, x, np64(inp["target"])


def make_layer(wl: W.Workload, inp: dict, device="cuda", group_score="top2_sum"):
    from sparse_mixture_experts_softmax_gb300.layer import MoELayer
    lp = wl.dtype == "bf16"
    return MoELayer(wl.T, wl.D, wl.F, wl.E, wl.k, wl.act, wl.score, wl.dtype, wl.has_bias,
                    wl.aux_alpha, inp["w_gate"], inp["w1"], inp["w2"], w3=inp["w3"],
                    b1=inp["b1"], b2=inp["b2"], logit_bias=inp["logit_bias"],
                    n_groups=wl.n_groups, topk_groups=wl.topk_groups, group_score=group_score,
                    w1_lp=inp.get("w1_bf16") if lp else None,
                    w3_lp=inp.get("w3_bf16") if lp else None,
                    w2_lp=inp.get("w2_bf16") if lp else None, device=device,
                    corr_bias=inp.get("corr_bias"), n_shared=wl.n_shared, ws1=inp.get("ws1"),
                    ws3=inp.get("ws3"), ws2=inp.get("ws2"), capacity_factor=wl.capacity_factor)


def device_x(wl: W.Workload, inp: dict, device="cuda"):
    return (inp["x_bf16"] if wl.dtype == "bf16" else inp["x"]).to(device).contiguous()


def rel_err(a, b) -> float:
    """max |a - b| / max |b| over a tensor (0 when both are all zero)."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.max(np.abs(b)) if b.size else 0.0
    num = np.max(np.abs(a - b)) if b.size else 0.0
    if den == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return float(num / den)


def assert_close(name, got, want, tol):
    err = rel_err(got, want)
    assert err <= tol, f"{name}: max-norm relative error {err:.3e} > {tol:.1e}"
    return err


def validated_relu_decisions(cfg: O.OracleConfig, st: dict, w: dict, h_kernel) -> int:
    """The ReLU derivative 1[h > 0] is a decision taken in floating point: a
    pre-activation within accumulation error of zero can fall on the kernel's
    side of zero differently from the float64 one.  Where the signs of the
    kernel's stored H (expert-major rows, the layer dtype) and the oracle's
    differ, check that the oracle's value lies within the fp32 accumulation
    error bound of zero, then let the oracle's backward take the kernel's
    decision (h set to a signed tiny value there; the forward values already
    computed are unchanged).  The bound: a sum of D products in fp32 (exact
    products of bf16 operands, or fused multiply-adds of fp32 ones) is within
    D u sum |x w| of its exact value, u = 2^-24; it is doubled for an adder
    that keeps one guard bit fewer (the tensor cores' accumulation order is
    not the oracle's), and the bias add is one more term: (D + 1) 2^-23
    (sum |x w| + |b|).  Returns the number of decisions taken from the
    kernel."""
    if cfg.act != "relu":
        return 0
    hk = np.asarray(h_kernel, dtype=np.float64)
    taken = 0
    for e in range(cfg.E):
        lo, hi = int(st["offsets"][e]), int(st["offsets"][e + 1])
        if hi == lo:
            continue
        fe = st["experts"][e]
        h64 = fe["h"]
        differ = (hk[lo:hi] > 0.0) != (h64 > 0.0)
        if not differ.any():
            continue
        scale = np.abs(st["xe"][lo:hi]) @ np.abs(w["w1"][e]).T
        if cfg.has_bias:
            scale = scale + np.abs(w["b1"][e])
        bound = (cfg.D + 1) * 2.0 ** -23 * scale[differ]
        assert np.all(np.abs(h64[differ]) <= bound), \
            f"expert {e}: ReLU decisions differ beyond rounding of a zero pre-activation"
        h_new = h64.copy()
        h_new[differ] = np.where(hk[lo:hi][differ] > 0.0, 1e-300, -1e-300)
        fe["h"] = h_new
        taken += int(differ.sum())
    return taken


def check_routing_exact(cfg: O.OracleConfig, r: dict, corr_bias=None):
    """Given the GPU's own fp32 scores, the oracle's selection and dispatch must
    reproduce idx, counts, offsets and both slot maps bit for bit.  A
    correction bias enters the keys as float32, the kernel's precision."""
    scores = r["scores"].cpu().numpy()            # float32, the kernel's precision
    idx_gpu = r["idx"].cpu().numpy()
    cb = None if corr_bias is None else corr_bias.detach().float().cpu().numpy()
    idx_o = O.route(cfg, scores, cb)
    np.testing.assert_array_equal(idx_gpu, idx_o)
    counts, offsets, src_tok, _, slot_of = O.dispatch(idx_gpu, cfg.E, O.expert_capacity(cfg))
    np.testing.assert_array_equal(r["counts"].cpu().numpy(), counts)
    np.testing.assert_array_equal(r["offsets"].cpu().numpy(), offsets)
    R = int(offsets[-1])   # kept rows (all T k of them without a capacity)
    np.testing.assert_array_equal(r["src_tok"].cpu().numpy()[:R], src_tok)
    np.testing.assert_array_equal(r["slot_of"].cpu().numpy(), slot_of)
    # gates: renormalised selected scores, in the kernel's fp32
    g = O.renormalize(scores.astype(np.float64), idx_gpu)
    assert rel_err(r["gate"].cpu().numpy(), g) <= 1e-6


def validated_routing(cfg: O.OracleConfig, scores64: np.ndarray, idx_gpu: np.ndarray,
                      margin_tol: float = 1e-5, corr_bias=None) -> np.ndarray:
    """Routing for the oracle's float values: its own fp64 selection, except on
    tokens where fp64 and the GPU's fp32 disagree AND the fp64 selection keys
    (scores, plus the correction bias if any) of the two choices lie within
    ``margin_tol`` of each other (a near-tie that rounding may legitimately
    flip).  Any other disagreement fails."""
    idx_o = O.route(cfg, scores64, corr_bias)
    keys = O.selection_keys(scores64, corr_bias)
    bad = np.nonzero(np.any(idx_o != idx_gpu, axis=1))[0]
    for t in bad:
        a = np.sort(keys[t, idx_o[t]])
        b = np.sort(keys[t, idx_gpu[t]])
        assert np.max(np.abs(a - b)) <= margin_tol * max(1.0, np.max(np.abs(keys[t]))), \
            f"token {t}: GPU routing {idx_gpu[t]} vs oracle {idx_o[t]} is not a near-tie"
    out = idx_o.copy()
    out[bad] = idx_gpu[bad]
    return out
