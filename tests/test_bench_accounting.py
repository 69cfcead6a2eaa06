"""bench.py's accounting, checked on the CPU against independent derivations.
These are the FLOPs and algorithmic bytes its roofline fractions divide by,
and the clock record it attaches to a measurement."""

from __future__ import annotations

import dataclasses

import bench
import workloads as W


def _gemm_flops_by_launch(wl: W.Workload, rows: int) -> float:
    """2 M N K summed over the expert GEMMs one training step launches,
    from each GEMM's operand shapes."""
    D, F = wl.D, wl.F
    f = 0.0
    if wl.act == "swiglu":
        f += 2 * rows * D * (2 * F)   # up: X_e [rows, D] x [W1; W3]^T -> H1, H3
    else:
        f += 2 * rows * D * F         # up: X_e W1^T -> H
    f += 2 * rows * F * D             # down: A W2^T -> Y_e
    f += 2 * rows * D * F             # dA = dY_e W2
    f += 2 * F * rows * D             # dW2 = dY_e^T A (ragged K = rows)
    if wl.act == "swiglu":
        f += 2 * rows * (2 * F) * D   # dX_e = dH1 W1 + dH3 W3
        f += 2 * 2 * F * rows * D     # dW1, dW3
    else:
        f += 2 * rows * F * D         # dX_e = dH W1
        f += 2 * F * rows * D         # dW1
    return f


def test_expert_flops_match_the_step_gemms():
    for name in ("tiny", "dense_f32", "dense_bf16", "grouped", "skewed", "large"):
        wl = W.WORKLOADS[name]
        assert bench.expert_flops_per_step(wl) == _gemm_flops_by_launch(wl, wl.R), name
        # a capacity: only the kept rows count
        assert bench.expert_flops_per_step(wl, 1000) == _gemm_flops_by_launch(wl, 1000), name
    # the large layer: 18 D F R = 79.16 TFLOP per step
    wl = W.WORKLOADS["large"]
    assert abs(bench.expert_flops_per_step(wl) - 79.164837199872e12) < 1.0


def test_shared_and_router_flops():
    wl = dataclasses.replace(W.WORKLOADS["large"], n_shared=1)
    Fs = wl.n_shared * wl.F
    fwd = 2 * wl.T * wl.D * Fs * 3          # Ws1, Ws3, Ws2 over all T tokens
    assert bench.shared_flops_per_step(wl) == 3 * fwd
    # logits, dW_g and the router dX: three T x D x E products
    assert bench.router_flops_per_step(wl) == 3 * 2 * wl.T * wl.D * wl.E


def test_hbm_bytes_from_tensor_sizes():
    for name in ("dense_f32", "grouped", "large"):
        wl = W.WORKLOADS[name]
        es = 2 if wl.dtype == "bf16" else 4
        T, D, R = wl.T, wl.D, wl.R
        x, rows, y32 = T * D * es, R * D * es, T * D * 4
        b = bench.hbm_bytes(wl)
        assert b["gather"] == x + rows                       # X read once, X_e written
        assert b["combine_fused"] == rows + y32 + rows       # Y_e, target in; dY_e out
        assert b["combine_loss"] == rows + y32 + y32         # Y_e, target in; dY out
        assert b["combine_bwd"] == y32 + rows + rows         # dY, Y_e in; dY_e out
    # the stand-alone SGD: 12 bytes per parameter (master and gradient read,
    # master written); bf16 layers keep only the router weight and biases here
    wl = W.WORKLOADS["dense_f32"]
    n = wl.E * wl.D + wl.E * (wl.F + wl.D) + 2 * wl.E * wl.D * wl.F
    assert bench.hbm_bytes(wl)["sgd"] == 12 * n
    wl = W.WORKLOADS["large"]
    assert bench.hbm_bytes(wl)["sgd"] == 12 * wl.E * wl.D


class _DoneProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_record_parsing():
    s = bench.ClockSampler(0)
    s.proc = _DoneProc()
    s.lines = [
        "1605, 2070, 1203.5, 0x4, Not Active, Not Active, Not Active, Active",
        "1680, 2070, 1350.1, 0x4, Not Active, Not Active, Not Active, Active",
        "1650, 2070, 1300.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "[N/A], [N/A], [N/A], [N/A], [N/A], [N/A], [N/A], [N/A]",   # ignored
        "garbage",                                                  # ignored
    ]
    rec = s.stop()
    assert rec["sm_mhz"] == 1650 and rec["sm_max_mhz"] == 2070
    assert rec["reasons"] == ["sw_power_cap"]
    s2 = bench.ClockSampler(0)
    s2.proc = _DoneProc()
    s2.lines = ["1500, 2070, 900, 0x8, Active, Not Active, Active, Not Active"]
    assert sorted(s2.stop()["reasons"]) == ["hw_slowdown", "sw_thermal_slowdown"]


def test_per_launch_flops_sum_to_the_step():
    """The per-launch split the bench reports adds up to the step's expert
    FLOPs, and each launch carries 2 M N K of its own operand shapes."""
    for name in ("tiny", "dense_f32", "dense_bf16", "grouped", "skewed", "large"):
        wl = W.WORKLOADS[name]
        per = bench.gemm_launch_flops(wl, 1234)
        assert abs(sum(per.values()) - bench.expert_flops_per_step(wl, 1234)) < 1e-6 * sum(per.values())
    wl = W.WORKLOADS["large"]
    per = bench.gemm_launch_flops(wl)
    R, D, F = wl.R, wl.D, wl.F
    assert per["gemm_up"] == 2 * R * D * (2 * F)       # [R, D] x [2F, D]^T
    assert per["gemm_dw1"] == 2 * F * D * R            # [F, R] x [R, D]
    assert per["gemm_dxe"] == 2 * R * (2 * F) * D      # [R, 2F] x [2F, D]


def test_scatter_back_bytes():
    wl = W.WORKLOADS["large"]
    # dXe [R, D] bf16 read; dX [T, D] fp32 read (router term) and written
    assert bench.hbm_bytes(wl)["scatter_back"] == wl.R * wl.D * 2 + 2 * wl.T * wl.D * 4


def test_cpu_baseline_extrapolation():
    """Per-token time scales with the tokens, SGD with the experts: a sample
    of 100 tokens over 16 of 128 experts taking 2 s + 0.5 s of SGD stands for
    a 65536-token step of 2 * 655.36 + 0.5 * 8 seconds."""
    wl = W.WORKLOADS["large"]
    rate = bench.extrapolated_rate(wl, 100, 16, 2.0, 0.5)
    assert abs(rate - 65536 / (2.0 * 655.36 + 0.5 * 8)) < 1e-9
