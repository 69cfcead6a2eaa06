"""Element-by-element parity at the per-expert shape of the large layer's
timed step: D = 4096, F = 2048, k = 8, SwiGLU, bf16 with fp32 masters, on
4096 tokens over 8 experts (every expert then holds 4096 rows, the M / K of
every expert GEMM of the 65536-token, 128-expert step) and over 16 experts
(ragged segments around 2048 rows).

Against the float64 oracle, in full: y, dX, dlogits, dW_g, every dW1, dW3,
dW2 (each expert on its own as well as the whole tensor), every expert's SGD
step theta_1 - theta_0 against -lr * grad, every bf16 working copy, and the
two losses.  Course "Trainable MoE in CUDA", Parts 5-7; the article's
"Design evidence that can falsify the implementation".
"""

import dataclasses

import numpy as np
import pytest
import torch

import workloads as W
from sparse_mixture_experts_softmax_gb300 import binding as B
from tests.moe_cases import assert_close, np64
from tests.test_gpu_parity import _one_step_parity

pytestmark = pytest.mark.gpu
TOL = 2e-2


@pytest.mark.parametrize("E", [8, 16])
def test_large_layer_expert_shape_in_full(E):
    wl = dataclasses.replace(W.WORKLOADS["large"], name=f"large_T4096_E{E}", T=4096, E=E)
    keep = {}
    errs, layer, inp = _one_step_parity(wl, keep=keep)
    st, g, master = keep["st"], keep["g"], keep["master"]
    errs["y"] = assert_close("y", np64(keep["y"]), st["y"], TOL)
    dlogits = torch.empty(wl.T, wl.E, device="cuda")
    B.moe_get_intermediates(layer.cfg, layer.workspace, dlogits=dlogits)
    torch.cuda.synchronize()
    errs["dlogits"] = assert_close("dlogits", np64(dlogits), g["dlogits"], TOL)
    rows = np.diff(st["offsets"])
    per_expert = {}
    for key in ("w1", "w3", "w2"):
        got = np64(getattr(layer, "d" + key))
        new = np64(getattr(layer, key))
        worst_g = worst_s = 0.0
        for e in range(wl.E):
            if rows[e] == 0:
                assert np.all(got[e] == 0.0), (key, e)
                continue
            worst_g = max(worst_g, assert_close(f"d{key}[{e}]", got[e], g["d" + key][e], TOL))
            # the step of expert e alone: theta_1 - theta_0 against -lr * grad,
            # widened by half an fp32 ulp of |theta| (the rounding of theta_1)
            want = -wl.lr * g["d" + key][e]
            scale = np.max(np.abs(want))
            tol = TOL + 2.0 ** -24 * np.max(np.abs(master[key][e])) / scale
            worst_s = max(worst_s, assert_close(f"step {key}[{e}]", new[e] - master[key][e],
                                                want, tol))
        per_expert["d" + key] = worst_g
        per_expert["step " + key] = worst_s
    print(f"\n{wl.name}: rows per expert {rows.tolist()}")
    print("  whole tensors: " + ", ".join(f"{k}={v:.2e}" for k, v in sorted(errs.items())))
    print("  worst expert:  " + ", ".join(f"{k}={v:.2e}" for k, v in sorted(per_expert.items())))
    assert max(errs.values()) <= TOL
    del layer, inp
    torch.cuda.empty_cache()
