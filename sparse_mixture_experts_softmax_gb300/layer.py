"""Device-buffer owner for one MoE layer, on top of the ctypes binding.

Allocates (through torch) the fp32 master parameters, the bf16 working copies,
the gradient buffers and the workspace, and calls the C ABI.  It computes
nothing itself.
"""

from __future__ import annotations

from typing import Optional

import torch

from . import binding as B


class MoELayer:
    def __init__(self, T, D, F, E, k, act, score, dtype, has_bias, aux_alpha, w_gate, w1, w2,
                 w3=None, b1=None, b2=None, logit_bias=None, n_groups=1, topk_groups=1,
                 group_score="top2_sum", w1_lp=None, w3_lp=None, w2_lp=None, device="cuda",
                 corr_bias=None, n_shared=0, ws1=None, ws3=None, ws2=None, capacity_factor=0.0,
                 store_grads=True):
        """store_grads=False: training steps pass NULL gradient buffers (the
        step still applies every gradient; bf16 layers then skip storing the
        expert weights' fp32 gradients) and no gradient tensors are
        allocated; ``backward`` is then unavailable."""
        self.device = torch.device(device)
        self.dtype = dtype
        self.cfg = B.make_config(T, D, F, E, k, act=act, score=score, n_groups=n_groups,
                                 topk_groups=topk_groups, group_score=group_score, dtype=dtype,
                                 has_bias=has_bias, aux_alpha=aux_alpha, n_shared=n_shared,
                                 capacity_factor=capacity_factor)
        dev = self.device

        def f32(t):
            return None if t is None else t.detach().to(dev, torch.float32).contiguous().clone()

        self.w_gate, self.w1, self.w2, self.w3 = f32(w_gate), f32(w1), f32(w2), f32(w3)
        self.b1, self.b2, self.logit_bias = f32(b1), f32(b2), f32(logit_bias)
        self.corr_bias = f32(corr_bias)   # selection-only routing bias (never trained)
        # shared-expert branch: fp32 masters and (bf16 layers) working copies
        self.ws1, self.ws3, self.ws2 = f32(ws1), f32(ws3), f32(ws2)
        if dtype == "bf16":
            def lp(given, master):
                if master is None:
                    return None
                src = given if given is not None else master
                return src.detach().to(dev, torch.bfloat16).contiguous().clone()
            self.w1_lp, self.w2_lp, self.w3_lp = lp(w1_lp, self.w1), lp(w2_lp, self.w2), lp(w3_lp, self.w3)
            self.ws1_lp, self.ws3_lp, self.ws2_lp = (lp(None, self.ws1), lp(None, self.ws3),
                                                     lp(None, self.ws2))
        else:
            self.w1_lp = self.w2_lp = self.w3_lp = None
            self.ws1_lp = self.ws3_lp = self.ws2_lp = None
        z = lambda t: None if t is None or not store_grads else torch.zeros_like(t)  # noqa: E731
        self.dw_gate, self.dw1, self.dw2, self.dw3 = z(self.w_gate), z(self.w1), z(self.w2), z(self.w3)
        self.db1, self.db2 = z(self.b1), z(self.b2)
        self.dws1, self.dws3, self.dws2 = z(self.ws1), z(self.ws3), z(self.ws2)
        self.grads = B.make_grads(self.dw_gate, self.dw1, self.dw2, self.dw3, self.db1, self.db2,
                                  self.dws1, self.dws3, self.dws2)
        self.ws_bytes = B.moe_workspace_size(self.cfg)
        if self.ws_bytes == 0:
            raise B.MoEError("moe_workspace_size", B.MOE_ERR_INVALID_ARG, "invalid configuration")
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.d_loss = torch.zeros(2, dtype=torch.float32, device=dev)

    # expert weights in the compute dtype (bf16 copies for bf16 layers)
    def weights(self) -> B.moe_weights:
        lp = self.dtype == "bf16"
        return B.make_weights(self.w_gate, self.w1_lp if lp else self.w1,
                              self.w2_lp if lp else self.w2, self.w3_lp if lp else self.w3,
                              self.b1, self.b2, self.logit_bias, self.corr_bias,
                              self.ws1_lp if lp else self.ws1, self.ws3_lp if lp else self.ws3,
                              self.ws2_lp if lp else self.ws2)

    def params(self) -> B.moe_params:
        return B.make_params(self.w_gate, self.w1, self.w2, self.grads, w3=self.w3, b1=self.b1,
                             b2=self.b2, w1_lp=self.w1_lp, w3_lp=self.w3_lp, w2_lp=self.w2_lp,
                             logit_bias=self.logit_bias, corr_bias=self.corr_bias,
                             ws1=self.ws1, ws3=self.ws3, ws2=self.ws2, ws1_lp=self.ws1_lp,
                             ws3_lp=self.ws3_lp, ws2_lp=self.ws2_lp)

    def forward(self, x: torch.Tensor, y: Optional[torch.Tensor] = None) -> torch.Tensor:
        if y is None:
            y = torch.empty(self.cfg.T, self.cfg.D, dtype=torch.float32, device=self.device)
        B.moe_forward(self.cfg, self.weights(), x, y, self.workspace)
        return y

    def backward(self, x: torch.Tensor, dy: torch.Tensor, dx: Optional[torch.Tensor] = None):
        if self.dw_gate is None:
            raise ValueError("this layer was built with store_grads=False: no gradient buffers")
        B.moe_backward(self.cfg, self.weights(), x, dy, self.grads, dx, self.workspace)
        return dx

    def train_step(self, x, target, lr, dx: Optional[torch.Tensor] = None) -> torch.Tensor:
        B.moe_train_step(self.cfg, self.params(), x, target, lr, self.d_loss, self.workspace, dx=dx)
        return self.d_loss

    def grad_dict(self) -> dict:
        return dict(dw_gate=self.dw_gate, dw1=self.dw1, dw2=self.dw2, dw3=self.dw3,
                    db1=self.db1, db2=self.db2, dws1=self.dws1, dws3=self.dws3, dws2=self.dws2)

    def param_dict(self) -> dict:
        return dict(w_gate=self.w_gate, w1=self.w1, w2=self.w2, w3=self.w3, b1=self.b1,
                    b2=self.b2, ws1=self.ws1, ws3=self.ws3, ws2=self.ws2)

    def routing(self) -> dict:
        c = self.cfg
        dev = self.device
        R = c.T * c.k
        out = dict(scores=torch.empty(c.T, c.E, device=dev),
                   idx=torch.empty(c.T, c.k, dtype=torch.int32, device=dev),
                   gate=torch.empty(c.T, c.k, device=dev),
                   counts=torch.empty(c.E, dtype=torch.int32, device=dev),
                   offsets=torch.empty(c.E + 1, dtype=torch.int32, device=dev),
                   src_tok=torch.empty(max(R, 1), dtype=torch.int32, device=dev),
                   slot_of=torch.empty(c.T, c.k, dtype=torch.int32, device=dev))
        B.moe_get_routing(c, self.workspace, **out)
        return out

    def hidden(self) -> dict:
        """The last forward's expert pre-activations [R, F] in the layer dtype:
        h1 (H, or H1 for SwiGLU) and h3 (SwiGLU only)."""
        c = self.cfg
        R = max(c.T * c.k, 1)
        dt = torch.bfloat16 if self.dtype == "bf16" else torch.float32
        h1 = torch.empty(R, c.F, dtype=dt, device=self.device)
        h3 = (torch.empty(R, c.F, dtype=dt, device=self.device)
              if c.act == B.ACT["swiglu"] else None)
        B.moe_get_hidden(c, self.workspace, h1=h1, h3=h3)
        return dict(h1=h1, h3=h3)
