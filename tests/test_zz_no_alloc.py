"""The workspace-free dispatch entry point (moe_dispatch_noalloc) against the
dispatch moe_forward performs with a caller workspace.

It serves callers that may not allocate device memory when they route (for
instance during CUDA graph capture); its scratch is a fixed array inside the
library.  This file is collected last so that a failure here cannot hide the
other tests in a run that stops at the first failure.
"""

import pytest
import torch

import workloads as W
from sparse_mixture_experts_softmax_gb300 import binding as B
from tests.moe_cases import device_x, make_layer

pytestmark = pytest.mark.gpu


def _reference_routing(name, T, seed):
    wl = W.WORKLOADS[name].with_tokens(T)
    inp = W.make_inputs(wl, seed=seed, with_target=False)
    inp["target"] = None
    layer = make_layer(wl, inp)
    layer.forward(device_x(wl, inp))
    torch.cuda.synchronize()
    return layer.cfg, layer.routing()


def _noalloc(cfg, idx):
    R = cfg.T * cfg.k
    out = dict(counts=torch.full((cfg.E,), -1, dtype=torch.int32, device="cuda"),
               offsets=torch.full((cfg.E + 1,), -1, dtype=torch.int32, device="cuda"),
               src_tok=torch.full((max(R, 1),), -1, dtype=torch.int32, device="cuda"),
               slot_of=torch.full((cfg.T, cfg.k), -1, dtype=torch.int32, device="cuda"))
    B.moe_dispatch_noalloc(cfg, idx, **out)
    torch.cuda.synchronize()
    return out


def test_noalloc_dispatch_matches_workspace_dispatch_twice():
    # two different routings back to back: the second call must not see the
    # first call's scratch contents
    for name, T, seed in (("skewed", 3000, 1), ("grouped", 1111, 2), ("skewed", 3000, 1)):
        cfg, ref = _reference_routing(name, T, seed)
        got = _noalloc(cfg, ref["idx"])
        R = cfg.T * cfg.k
        assert torch.equal(got["counts"], ref["counts"])
        assert torch.equal(got["offsets"], ref["offsets"])
        assert torch.equal(got["src_tok"][:R], ref["src_tok"][:R])
        assert torch.equal(got["slot_of"], ref["slot_of"])


def test_noalloc_dispatch_rejects_too_many_rows():
    cfg = B.make_config(T=B.MOE_NOALLOC_MAX_ROUTED // 8 + 1, D=64, F=64, E=64, k=8,
                        act="swiglu", has_bias=False, dtype="bf16")
    with pytest.raises(B.MoEError) as ei:
        B.moe_dispatch_noalloc(cfg, None, None, None, None, None)
    assert ei.value.status == B.MOE_ERR_UNSUPPORTED
