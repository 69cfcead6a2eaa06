"""The workspace-free dispatch entry point (moe_dispatch_noalloc) against the
oracle's dispatch (per-expert counts, exclusive-scan offsets, the stable slot
map), through the C ABI.

It serves callers that may not allocate device memory when they route (for
instance during CUDA graph capture, or inside a runtime that owns all device
memory); its scratch is a fixed array inside the library, shared by every
call.  Consecutive calls with different routings check that no call sees the
previous call's scratch contents.  This file is collected last so that a
failure here cannot hide the other tests in a run that stops at the first
failure.
"""

import numpy as np
import pytest
import torch

import workloads as W
from oracle import moe_oracle as O
from sparse_mixture_experts_softmax_gb300 import binding as B
from tests.moe_cases import device_x, make_layer, oracle_config

pytestmark = pytest.mark.gpu


def _routing(name, T, seed, capacity_factor=None):
    """A real routing of a seeded workload (idx from the library's router)."""
    import dataclasses
    wl = W.WORKLOADS[name].with_tokens(T)
    if capacity_factor is not None:
        wl = dataclasses.replace(wl, capacity_factor=capacity_factor)
    inp = W.make_inputs(wl, seed=seed, with_target=False)
    inp["target"] = None
    layer = make_layer(wl, inp)
    layer.forward(device_x(wl, inp))
    torch.cuda.synchronize()
    return wl, layer.cfg, layer.routing()["idx"]


def _noalloc(cfg, idx):
    R = cfg.T * cfg.k
    out = dict(counts=torch.full((cfg.E,), -7, dtype=torch.int32, device="cuda"),
               offsets=torch.full((cfg.E + 1,), -7, dtype=torch.int32, device="cuda"),
               src_tok=torch.full((max(R, 1),), -7, dtype=torch.int32, device="cuda"),
               slot_of=torch.full((max(cfg.T, 1), cfg.k), -7, dtype=torch.int32, device="cuda"))
    B.moe_dispatch_noalloc(cfg, idx, **out)
    torch.cuda.synchronize()
    return {k_: v.cpu().numpy() for k_, v in out.items()}


def _check_against_oracle(wl, got, idx_np):
    counts, offsets, src_tok, _, slot_of = O.dispatch(idx_np, wl.E,
                                                     O.expert_capacity(oracle_config(wl)))
    np.testing.assert_array_equal(got["counts"], counts)
    np.testing.assert_array_equal(got["offsets"], offsets)
    kept = int(offsets[-1])
    np.testing.assert_array_equal(got["src_tok"][:kept], src_tok)
    np.testing.assert_array_equal(got["slot_of"][:wl.T], slot_of)
    return kept


def test_noalloc_dispatch_matches_oracle_on_consecutive_calls():
    # different routings back to back (a skewed one with empty experts, a
    # grouped one, the skewed one again): each call starts from the previous
    # call's scratch contents
    for name, T, seed in (("skewed", 3000, 1), ("grouped", 1111, 2), ("skewed", 3000, 1)):
        wl, cfg, idx = _routing(name, T, seed)
        got = _noalloc(cfg, idx)
        kept = _check_against_oracle(wl, got, idx.cpu().numpy())
        assert kept == wl.T * wl.k


def test_noalloc_dispatch_with_expert_capacity():
    """Each expert keeps its first C = ceil(cf T k / E) assignments in token
    order; the rest get slot -1; counts stay the routed (pre-drop) counts."""
    for name, T, cf in (("skewed", 2000, 1.25), ("dense_f32", 3000, 0.75)):
        wl, cfg, idx = _routing(name, T, 3, capacity_factor=cf)
        got = _noalloc(cfg, idx)
        kept = _check_against_oracle(wl, got, idx.cpu().numpy())
        dropped = int((got["slot_of"][:wl.T] < 0).sum())
        assert dropped > 0 and kept + dropped == wl.T * wl.k


def test_noalloc_dispatch_empty_tokens():
    """T = 0: every count and offset is zero, nothing else is written."""
    cfg = B.make_config(T=0, D=64, F=64, E=16, k=4, act="swiglu", has_bias=False, dtype="bf16")
    got = _noalloc(cfg, None)
    assert np.all(got["counts"] == 0) and np.all(got["offsets"] == 0)
    assert np.all(got["src_tok"] == -7) and np.all(got["slot_of"] == -7)


def test_noalloc_dispatch_out_of_range_expert_id():
    """A token whose expert ids lie outside [0, E) is not counted and gets
    slot -1; the other tokens dispatch as if it were absent."""
    wl, cfg, idx = _routing("grouped", 900, 4)
    bad = idx.clone()
    bad[-1] = torch.tensor([wl.E + j for j in range(wl.k)], dtype=torch.int32)
    got = _noalloc(cfg, bad)
    idx_np = idx.cpu().numpy()[:-1]
    counts, offsets, src_tok, _, slot_of = O.dispatch(idx_np, wl.E)
    np.testing.assert_array_equal(got["counts"], counts)
    np.testing.assert_array_equal(got["offsets"], offsets)
    np.testing.assert_array_equal(got["src_tok"][:int(offsets[-1])], src_tok)
    np.testing.assert_array_equal(got["slot_of"][:-1], slot_of)
    assert np.all(got["slot_of"][-1] == -1)


def test_noalloc_dispatch_rejects_bad_requests():
    cfg = B.make_config(T=B.MOE_NOALLOC_MAX_ROUTED // 8 + 1, D=64, F=64, E=64, k=8,
                        act="swiglu", has_bias=False, dtype="bf16")
    with pytest.raises(B.MoEError) as ei:
        B.moe_dispatch_noalloc(cfg, None, None, None, None, None)
    assert ei.value.status == B.MOE_ERR_UNSUPPORTED
    for cf in (float("nan"), -1.0):
        cfg = B.make_config(T=8, D=64, F=64, E=16, k=2, act="swiglu", has_bias=False,
                            dtype="bf16", capacity_factor=cf)
        with pytest.raises(B.MoEError) as ei:
            B.moe_dispatch_noalloc(cfg, None, None, None, None, None)
        assert ei.value.status == B.MOE_ERR_INVALID_ARG
