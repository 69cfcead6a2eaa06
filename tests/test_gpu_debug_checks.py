"""The MOE_DEBUG variant of the library (libmoe_gb300_debug.so): device-side
checks of every routing index before it is dereferenced (the course
article's call for race and out-of-bounds checks, with compute-sanitizer not
available).

* On valid routing (a capacity that drops assignments included) the debug
  library reports nothing and gives the release library's bits.
* With routing state corrupted on purpose (moe_debug_poke_routing: an
  expert-major slot past the routed rows, a negative slot, an expert id past
  E), the checked kernels skip those entries and record MOE_ERR_INVALID_ARG
  in the workspace status word; a guard band on both sides of the workspace
  keeps its bytes, and every token the corruption does not touch gets the
  release library's dL/dx bit for bit.  The corrupt values are chosen to lie
  inside the workspace allocation, so even a missing check would not leave
  the caller's memory.
"""

import dataclasses

import numpy as np
import pytest
import torch

import workloads as W
from sparse_mixture_experts_softmax_gb300 import binding as B
from tests.moe_cases import device_x, make_layer

pytestmark = pytest.mark.gpu

GUARD = 1 << 20


def _guarded(layer):
    """Move the layer's workspace into the middle of a larger buffer whose
    guard bands hold a known byte pattern."""
    buf = torch.full((layer.ws_bytes + 2 * GUARD,), 0x5A, dtype=torch.uint8, device="cuda")
    layer.workspace = buf[GUARD:GUARD + layer.ws_bytes]
    return buf


def _guards_intact(buf, n):
    return bool(torch.all(buf[:GUARD] == 0x5A)) and bool(torch.all(buf[GUARD + n:] == 0x5A))


def _workload(cf=0.0):
    return dataclasses.replace(W.WORKLOADS["dense_bf16"], name="dbg", T=300, D=256, F=128,
                               capacity_factor=cf)


def test_debug_library_is_the_checked_variant():
    assert B.moe_build_flags() == 0
    with B.use_library(debug=True):
        assert B.moe_build_flags() == B.MOE_BUILD_DEBUG_CHECKS
    assert B.moe_build_flags() == 0


@pytest.mark.parametrize("cf", [0.0, 0.75])
def test_valid_routing_reports_nothing_and_matches_release(cf):
    wl = _workload(cf)
    inp = W.make_inputs(wl, seed=3)
    x = device_x(wl, inp)
    dy = torch.randn(wl.T, wl.D, generator=torch.Generator().manual_seed(4)).cuda() * 1e-3
    rel = make_layer(wl, inp)
    y_rel = rel.forward(x).clone()
    dx_rel = rel.backward(x, dy, torch.empty_like(dy)).clone()
    with B.use_library(debug=True):
        dbg = make_layer(wl, inp)
        buf = _guarded(dbg)
        y = dbg.forward(x).clone()
        dx = dbg.backward(x, dy, torch.empty_like(dy))
        assert B.moe_device_status(dbg.cfg, dbg.workspace) == 0
    torch.cuda.synchronize()
    assert torch.equal(y, y_rel) and torch.equal(dx, dx_rel)
    for k_, v in rel.grad_dict().items():
        if v is not None:
            assert torch.equal(v, dbg.grad_dict()[k_]), k_
    assert _guards_intact(buf, dbg.ws_bytes)
    if cf > 0:
        assert int((rel.routing()["slot_of"] < 0).sum().item()) > 0   # drops were present


def test_corrupt_routing_is_skipped_and_reported():
    wl = _workload()
    inp = W.make_inputs(wl, seed=5)
    x = device_x(wl, inp)
    dy = torch.randn(wl.T, wl.D, generator=torch.Generator().manual_seed(6)).cuda() * 1e-3
    rel = make_layer(wl, inp)
    rel.forward(x)
    dx_rel = rel.backward(x, dy, torch.empty_like(dy)).clone()
    R = wl.T * wl.k
    t_slot_hi, t_slot_neg, t_idx = 17, 123, 250
    with B.use_library(debug=True):
        dbg = make_layer(wl, inp)
        buf = _guarded(dbg)
        dbg.forward(x)
        assert B.moe_device_status(dbg.cfg, dbg.workspace) == 0
        # built on the host: one slot past the routed rows, one below -1, one
        # expert id past E
        B.moe_debug_poke_routing(dbg.cfg, dbg.workspace, 1, t_slot_hi * wl.k + 0, R + 5)
        B.moe_debug_poke_routing(dbg.cfg, dbg.workspace, 1, t_slot_neg * wl.k + 1, -7)
        B.moe_debug_poke_routing(dbg.cfg, dbg.workspace, 0, t_idx * wl.k + 0, wl.E + 3)
        dx = dbg.backward(x, dy, torch.empty_like(dy))
        status = B.moe_device_status(dbg.cfg, dbg.workspace)
        assert status == B.MOE_ERR_INVALID_ARG
        # the next forward clears the status word and rebuilds the routing
        dbg.forward(x)
        dx2 = dbg.backward(x, dy, torch.empty_like(dy))
        assert B.moe_device_status(dbg.cfg, dbg.workspace) == 0
    torch.cuda.synchronize()
    assert _guards_intact(buf, dbg.ws_bytes)
    untouched = np.setdiff1d(np.arange(wl.T), [t_slot_hi, t_slot_neg, t_idx])
    assert torch.equal(dx[untouched], dx_rel[untouched])
    assert torch.equal(dx2, dx_rel)


def test_release_library_refuses_to_corrupt_its_state():
    wl = _workload()
    inp = W.make_inputs(wl, seed=5)
    layer = make_layer(wl, inp)
    with pytest.raises(B.MoEError) as ei:
        B.moe_debug_poke_routing(layer.cfg, layer.workspace, 1, 0, 10 ** 6)
    assert ei.value.status == B.MOE_ERR_UNSUPPORTED
