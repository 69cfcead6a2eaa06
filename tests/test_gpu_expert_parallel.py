"""The expert-parallel training step on one GPU: G ranks driven by one
process (``LocalTransport``), each rank with its own tokens, workspace and
local experts, every phase running the library's kernels through the C ABI.

"AI Infra Kernel Lab", "Project status" (expert parallelism over a variable
All-to-All) and "Numerical contracts" (unweighted rows dispatched, routing
weights applied after the outputs return to their source rank, uneven and
empty token shards, the backward through both exchanges).

Checked against
* the float64 oracle of the WHOLE layer on the concatenation of the ranks'
  tokens: both losses, dL/dx of every token, dW_g (summed over the ranks), the
  local experts' gradients and SGD steps, the router's SGD step;
* the single-device training step of the same layer on the same tokens, bit
  for bit where the arithmetic is the same: every expert's updated fp32
  master and bf16 copy, and dL/dx (an owner holds an expert's rows in the
  single device's order).  The router's gradient is a sum over ranks here
  and over token chunks there, so W_g is compared within rounding.
"""

import dataclasses

import numpy as np
import pytest
import torch

import workloads as W
from oracle import moe_oracle as O
from sparse_mixture_experts_softmax_gb300 import expert_parallel as EP
from tests.moe_cases import (TOL, assert_close, device_x, make_layer, np64, oracle_config,
                             oracle_inputs, validated_routing)

pytestmark = pytest.mark.gpu

CASES = {
    # bf16 SwiGLU, softmax + aux, four ranks with uneven and empty shards,
    # gradients not stored (the fused SGD applies them)
    "swiglu_bf16_g4": (dataclasses.replace(W.WORKLOADS["large"], name="ep_swiglu", D=512, F=256,
                                           E=16, k=4, T=1028), (300, 0, 517, 211), False),
    # fp32 GELU experts with biases, two ranks
    "gelu_f32_g2": (dataclasses.replace(W.WORKLOADS["dense_f32"], name="ep_gelu", T=769),
                    (640, 129), True),
    # fp32 SwiGLU experts (GEMMs through the three-term split on the tensor
    # cores, two-pair dXe included), two ranks
    "swiglu_f32_g2": (dataclasses.replace(W.WORKLOADS["dense_f32"], name="ep_swiglu_f32",
                                          act="swiglu", has_bias=False, T=500), (300, 200), True),
    # grouped sigmoid routing over eight ranks (8 local experts each)
    "grouped_bf16_g8": (dataclasses.replace(W.WORKLOADS["grouped"], name="ep_grouped", D=256,
                                            F=128, T=900),
                        (200, 0, 130, 70, 0, 250, 150, 100), True),
    # k > 8: the separate combine and combine-backward kernels
    "swiglu_bf16_k10_g2": (dataclasses.replace(W.WORKLOADS["large"], name="ep_k10", D=256,
                                               F=128, E=16, k=10, T=177), (100, 77), True),
}


def _ranks(wl, inp, shards, store_grads):
    G = len(shards)
    return [EP.EPRank(r, G, shards[r], wl.T, wl.D, wl.F, wl.E, wl.k, wl.act, wl.score, wl.dtype,
                      wl.has_bias, wl.aux_alpha, inp["w_gate"], inp["w1"], inp["w2"],
                      w3=inp["w3"], b1=inp["b1"], b2=inp["b2"], logit_bias=inp["logit_bias"],
                      corr_bias=inp.get("corr_bias"), n_groups=wl.n_groups,
                      topk_groups=wl.topk_groups, store_grads=store_grads)
            for r in range(G)]


@pytest.mark.parametrize("name", sorted(CASES))
def test_expert_parallel_step(name):
    wl, shards, store = CASES[name]
    assert sum(shards) == wl.T
    G, L = len(shards), wl.E // len(shards)
    inp = W.make_inputs(wl, seed=21)
    tol = TOL[wl.dtype]
    x = device_x(wl, inp)
    tgt = inp["target"].cuda()
    cut = np.concatenate([[0], np.cumsum(shards)])
    xs = {r: x[cut[r]:cut[r + 1]].contiguous() for r in range(G)}
    ts = {r: tgt[cut[r]:cut[r + 1]].contiguous() for r in range(G)}
    dxs = {r: torch.empty(shards[r], wl.D, device="cuda") for r in range(G)}
    ranks = _ranks(wl, inp, shards, store)
    out = EP.train_step(ranks, EP.LocalTransport(G), xs, ts, wl.lr, dxs)
    torch.cuda.synchronize()
    assert sum(out["rows_received"].values()) == wl.T * wl.k
    assert all(int(rk.status.max().item()) == 0 for rk in ranks)

    # --- the single-device step on the same tokens
    layer = make_layer(wl, inp)
    dx1 = torch.empty(wl.T, wl.D, device="cuda")
    layer.train_step(x, tgt, wl.lr, dx=dx1)
    torch.cuda.synchronize()
    for key in ("w1", "w3", "w2", "b1", "b2"):
        ref = getattr(layer, key)
        if ref is None:
            continue
        got = torch.cat([getattr(rk, key) for rk in ranks])
        assert torch.equal(got, ref), key
        if wl.dtype == "bf16" and key in ("w1", "w3", "w2"):
            assert torch.equal(torch.cat([getattr(rk, key + "_lp") for rk in ranks]),
                               getattr(layer, key + "_lp")), key
    assert torch.equal(torch.cat([dxs[r] for r in range(G)]), dx1)
    for rk in ranks:
        assert torch.equal(rk.w_gate, ranks[0].w_gate)        # replicated router stays in step
    assert_close("w_gate vs single device", np64(ranks[0].w_gate), np64(layer.w_gate), 1e-6)
    loss1 = layer.d_loss.cpu().numpy()
    assert_close("mse vs single device", out["mse"], loss1[0], 1e-5)
    assert_close("aux vs single device", out["aux"], loss1[1], 1e-5)

    # --- the oracle of the whole layer
    cfg = oracle_config(wl)
    w_fwd, master, x64, t64 = oracle_inputs(wl, inp)
    idx_gpu = np.concatenate([rk.routing()["idx"].cpu().numpy() for rk in ranks])
    for rk in ranks:                      # each rank's routing, bit-exact given its scores
        rt = rk.routing()
        np.testing.assert_array_equal(rt["idx"].cpu().numpy(),
                                      O.route(cfg, rt["scores"].cpu().numpy(),
                                              w_fwd.get("corr_bias")))
    scores64 = O.router_scores(cfg, O.router_logits(x64, w_fwd["w_gate"], w_fwd["logit_bias"]))
    idx = validated_routing(cfg, scores64, idx_gpu, corr_bias=w_fwd.get("corr_bias"))
    st = O.forward(cfg, w_fwd, x64, idx)
    l_mse, aux, dy = O.losses(cfg, st, t64)
    g = O.backward(cfg, w_fwd, x64, st, dy)
    errs = {"mse": assert_close("mse", out["mse"], l_mse, tol),
            "aux": assert_close("aux", out["aux"], aux, tol),
            "dx": assert_close("dx", np64(torch.cat([dxs[r] for r in range(G)])), g["dx"], tol),
            "dw_gate": assert_close("dw_gate", np64(ranks[0].dw_gate), g["dw_gate"], tol)}
    for r, rk in enumerate(ranks):
        lo, hi = r * L, (r + 1) * L
        for key in ("w1", "w3", "w2", "b1", "b2"):
            if master.get(key) is None:
                continue
            want_step = -wl.lr * g["d" + key][lo:hi]
            step = np64(getattr(rk, key)) - master[key][lo:hi]
            scale = np.max(np.abs(want_step))
            if scale == 0:
                assert np.all(step == 0), (r, key)      # experts without rows stay put
                continue
            assert_close(f"step {key}@{r}", step, want_step,
                         tol + 2.0 ** -24 * np.max(np.abs(master[key][lo:hi])) / scale)
            grad = getattr(rk, "d" + key)
            if grad is not None:
                errs[f"d{key}@{r}"] = assert_close(f"d{key}@{r}", np64(grad),
                                                   g["d" + key][lo:hi], tol)
    want = master["w_gate"] - wl.lr * g["dw_gate"]
    assert_close("w_gate", np64(ranks[0].w_gate), want, tol)
    print(f"\n{name}: shards {shards}, rows received {out['rows_received']}; "
          + ", ".join(f"{k}={v:.2e}" for k, v in sorted(errs.items())))
