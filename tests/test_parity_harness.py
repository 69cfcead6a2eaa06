"""The parity harness's two validated floating-point decisions, checked on
the CPU against planted kernel outputs.

- ReLU derivatives: a sign flip at a pre-activation within rounding of zero
  is taken from the kernel, and changes the oracle's dH there only. A flip
  anywhere else fails.
- Routing: a selection that differs from the oracle's own only on near-tied
  (or exactly tied) keys is taken from the kernel. Any other difference fails.
"""

from __future__ import annotations

import numpy as np
import pytest

from oracle import moe_oracle as O
from tests.moe_cases import validated_relu_decisions, validated_routing


def _case():
    cfg = O.OracleConfig(T=24, D=16, F=8, E=3, k=2, act="relu", score="softmax",
                         has_bias=True, aux_alpha=0.0)
    rng = np.random.default_rng(5)
    w = dict(w_gate=rng.normal(0, 0.3, (3, 16)), w1=rng.normal(0, 0.3, (3, 8, 16)),
             w2=rng.normal(0, 0.3, (3, 16, 8)), w3=None, b1=rng.normal(0, 0.1, (3, 8)),
             b2=np.zeros((3, 16)))
    x = rng.normal(0, 1, (24, 16))
    return cfg, w, x


def _kernel_h(st):
    """The oracle's own H in expert-major rows: what an exact kernel would store."""
    R = int(st["offsets"][-1])
    h = np.zeros((R, 8))
    for e in range(3):
        lo, hi = int(st["offsets"][e]), int(st["offsets"][e + 1])
        h[lo:hi] = st["experts"][e]["h"]
    return h


def test_no_flip_takes_nothing():
    cfg, w, x = _case()
    st = O.forward(cfg, w, x)
    assert validated_relu_decisions(cfg, st, w, _kernel_h(st)) == 0


def test_flip_within_rounding_is_taken_from_the_kernel():
    cfg, w, x = _case()
    st = O.forward(cfg, w, x)
    lo = int(st["offsets"][1])
    # plant an exactly representable near-zero pre-activation in the oracle's
    # H of expert 1 (row 0, column 3), negative in float64 ...
    st["experts"][1]["h"][0, 3] = -1e-9
    hk = _kernel_h(st)
    hk[lo, 3] = 1e-9          # ... and positive in the kernel's
    dy = np.random.default_rng(6).normal(0, 1, (24, 16))
    g_before = O.backward(cfg, w, x, st, dy)
    assert validated_relu_decisions(cfg, st, w, hk) == 1
    assert st["experts"][1]["h"][0, 3] > 0
    g_after = O.backward(cfg, w, x, st, dy)
    # dW1 of expert 1 changes in row 3 only; the other experts are untouched
    diff = np.abs(g_after["dw1"] - g_before["dw1"]) > 0
    assert diff[1, 3].any() and not diff[1, :3].any() and not diff[1, 4:].any()
    assert not diff[0].any() and not diff[2].any()


def test_bound_grows_with_the_reduction_length():
    """A flip at |h| just inside (D + 1) 2^-23 sum |x w| is taken, just outside
    it fails: the bound is the fp32 accumulation error of a D-term sum."""
    cfg, w, x = _case()
    for factor, ok in ((0.9, True), (1.1, False)):
        st = O.forward(cfg, w, x)
        lo = int(st["offsets"][1])
        scale = np.abs(st["xe"][lo]) @ np.abs(w["w1"][1][3]) + abs(w["b1"][1][3])
        h = factor * (cfg.D + 1) * 2.0 ** -23 * scale
        st["experts"][1]["h"][0, 3] = -h
        hk = _kernel_h(st)
        hk[lo, 3] = h
        if ok:
            assert validated_relu_decisions(cfg, st, w, hk) == 1
        else:
            with pytest.raises(AssertionError):
                validated_relu_decisions(cfg, st, w, hk)


def test_flip_beyond_rounding_fails():
    cfg, w, x = _case()
    st = O.forward(cfg, w, x)
    hk = _kernel_h(st)
    e = next(e for e in range(3) if st["offsets"][e + 1] > st["offsets"][e])
    lo = int(st["offsets"][e])
    j = int(np.argmax(np.abs(st["experts"][e]["h"][0])))
    hk[lo, j] = -st["experts"][e]["h"][0, j]     # a clear sign error in the kernel
    with pytest.raises(AssertionError):
        validated_relu_decisions(cfg, st, w, hk)


# ------------------------------------------------------- validated routing ---
# The other floating-point decision the harness takes from the kernel: a
# routing that differs from the oracle's own only on near-ties of the keys.

def _route_case():
    cfg = O.OracleConfig(T=4, D=1, F=1, E=6, k=2, score="softmax")
    scores = np.array([[0.30, 0.25, 0.20, 0.10, 0.10, 0.05],
                       [0.20, 0.20, 0.20, 0.20, 0.10, 0.10],
                       [0.05, 0.40, 0.40 - 1e-9, 0.05, 0.05, 0.05],
                       [0.10, 0.10, 0.10, 0.10, 0.30, 0.30]])
    return cfg, scores


def test_identical_routing_is_the_oracles():
    cfg, s = _route_case()
    idx = O.route(cfg, s)
    np.testing.assert_array_equal(validated_routing(cfg, s, idx.copy()), idx)


def test_near_tie_flip_is_taken_from_the_kernel():
    cfg, s = _route_case()
    idx = O.route(cfg, s)
    assert list(idx[2]) == [1, 2]   # 0.40 ahead of 0.40 - 1e-9
    kernel = idx.copy()
    kernel[2] = [2, 1]              # rounding put the near-tied pair the other way round
    out = validated_routing(cfg, s, kernel)
    np.testing.assert_array_equal(out[2], [2, 1])
    np.testing.assert_array_equal(np.delete(out, 2, axis=0), np.delete(idx, 2, axis=0))
    # an exact tie broken the other way round is a near-tie too (distance 0)
    kernel = idx.copy()
    kernel[1] = [2, 3]              # 0.20 x 4: the oracle keeps 0, 1 (smaller ids)
    out = validated_routing(cfg, s, kernel)
    np.testing.assert_array_equal(out[1], [2, 3])


def test_routing_flip_beyond_rounding_fails():
    cfg, s = _route_case()
    idx = O.route(cfg, s)
    kernel = idx.copy()
    kernel[0] = [0, 3]              # 0.10 instead of 0.25: not a near-tie
    with pytest.raises(AssertionError):
        validated_routing(cfg, s, kernel)
