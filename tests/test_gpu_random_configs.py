"""Seeded random layer configurations within the library's limits, one
training step each on the GPU against the oracle.

The draws combine the options the named workloads test one at a time (and a
second set reaches toward the library's limits):
- fp32 or bf16;
- ReLU, GELU-tanh or SwiGLU experts, with or without biases;
- softmax or sigmoid scores;
- plain or group-limited top-k, with k up to 12 (past the fused combine);
- a correction bias, an expert capacity and shared experts;
- ragged token counts and widths.

Each case checks routing, counts, offsets and slots bit for bit. Losses, every
gradient, dX and the updated weights must match within the tolerance of the
expert dtype. The draws are fixed by a seed, so a failing case id names a
reproducible configuration.
"""

from __future__ import annotations

import numpy as np
import pytest

import workloads as W
from tests.test_gpu_parity import _one_step_parity

N_CASES = 32
MASTER_SEED = 20261202


def _divisors(n, hi):
    return [d for d in range(2, min(n, hi) + 1) if n % d == 0]


def draw_workload(i: int) -> W.Workload:
    rng = np.random.default_rng([MASTER_SEED, i])
    dtype = str(rng.choice(["f32", "bf16"], p=[0.35, 0.65]))
    act = str(rng.choice(["relu", "gelu_tanh", "swiglu"]))
    score = str(rng.choice(["softmax", "sigmoid"]))
    # bf16 layers need E % 8 == 0 (row alignment of the router's bf16 tensors)
    E = int(rng.choice([8, 16, 24, 32, 48, 64] if dtype == "bf16" else [3, 5, 8, 12, 16, 40]))
    n_groups = topk_groups = 1
    divs = _divisors(E, 32)
    if divs and rng.random() < 0.4:
        n_groups = int(rng.choice(divs))
        topk_groups = int(rng.integers(1, n_groups + 1))
    k_max = min(12, topk_groups * (E // n_groups))
    k = int(rng.integers(1, k_max + 1))
    T = int(rng.integers(1, 700))
    D = 8 * int(rng.integers(2, 48))
    F = 8 * int(rng.integers(2, 48))
    has_bias = act != "swiglu" and bool(rng.random() < 0.5)
    n_shared = int(rng.integers(1, 3)) if (act == "swiglu" and dtype == "bf16"
                                           and rng.random() < 0.3) else 0
    capacity_factor = float(rng.choice([0.0, 0.0, 0.75, 1.25]))
    corr_bias_scale = 0.1 if rng.random() < 0.3 else None
    aux_alpha = float(rng.choice([0.0, 0.01]))
    return W.Workload(name=f"random{i}", T=T, D=D, F=F, E=E, k=k, act=act, score=score,
                      n_groups=n_groups, topk_groups=topk_groups, has_bias=has_bias,
                      dtype=dtype, aux_alpha=aux_alpha, lr=0.01,
                      corr_bias_scale=corr_bias_scale, n_shared=n_shared,
                      capacity_factor=capacity_factor)


def _case_id(i):
    wl = draw_workload(i)
    opts = [wl.dtype, wl.act, wl.score, f"T{wl.T}", f"D{wl.D}", f"F{wl.F}", f"E{wl.E}",
            f"k{wl.k}"]
    if wl.n_groups > 1:
        opts.append(f"g{wl.n_groups}of{wl.topk_groups}")
    if wl.has_bias:
        opts.append("bias")
    if wl.n_shared:
        opts.append(f"shared{wl.n_shared}")
    if wl.capacity_factor:
        opts.append(f"cf{wl.capacity_factor}")
    if wl.corr_bias_scale:
        opts.append("cb")
    return "-".join(opts)


def test_draws_are_within_the_limits():
    for i in range(N_CASES):
        wl = draw_workload(i)
        assert wl.D % 8 == 0 and wl.F % 8 == 0 and 1 <= wl.k <= wl.E
        assert wl.E % wl.n_groups == 0 and wl.k <= wl.topk_groups * (wl.E // wl.n_groups)
        assert wl.dtype == "f32" or wl.E % 8 == 0
        assert not (wl.act == "swiglu" and wl.has_bias)
        assert not wl.n_shared or (wl.act == "swiglu" and wl.dtype == "bf16")


@pytest.mark.gpu
@pytest.mark.parametrize("i", range(N_CASES), ids=[_case_id(i) for i in range(N_CASES)])
def test_random_configuration_step(i):
    wl = draw_workload(i)
    errs, _, _ = _one_step_parity(wl, seed=100 + i)
    assert np.isfinite(max(errs.values()))


# Draws near the limits: E up to 256, k up to 32, D and F up to 1024, T up to
# 2048.  A cheap subset of one seed's draws is kept here (the oracle's cost
# grows with T k D F), each with the input seed it was validated with.
WIDE_SEED = 99
WIDE_CASES = (1, 4, 13, 18, 19, 24, 29, 37)


def draw_wide_workload(i: int) -> W.Workload:
    rng = np.random.default_rng([WIDE_SEED, i])
    dtype = str(rng.choice(["f32", "bf16"], p=[0.3, 0.7]))
    act = str(rng.choice(["relu", "gelu_tanh", "swiglu"]))
    score = str(rng.choice(["softmax", "sigmoid"]))
    E = int(rng.choice([64, 128, 192, 256] if dtype == "bf16" else [7, 33, 100, 256]))
    n_groups = topk_groups = 1
    divs = _divisors(E, 32)
    if divs and rng.random() < 0.4:
        n_groups = int(rng.choice(divs))
        topk_groups = int(rng.integers(1, n_groups + 1))
    k_max = min(32, topk_groups * (E // n_groups))
    k = int(rng.integers(1, k_max + 1))
    T = int(rng.integers(1, 2048))
    D = 8 * int(rng.integers(1, 129))
    F = 8 * int(rng.integers(1, 129))
    has_bias = act != "swiglu" and bool(rng.random() < 0.5)
    n_shared = int(rng.integers(1, 3)) if (act == "swiglu" and dtype == "bf16"
                                           and rng.random() < 0.3) else 0
    capacity_factor = float(rng.choice([0.0, 0.0, 0.5, 1.0, 2.0]))
    corr_bias_scale = 0.1 if rng.random() < 0.3 else None
    aux_alpha = float(rng.choice([0.0, 0.01]))
    return W.Workload(name=f"wide{i}", T=T, D=D, F=F, E=E, k=k, act=act, score=score,
                      n_groups=n_groups, topk_groups=topk_groups, has_bias=has_bias,
                      dtype=dtype, aux_alpha=aux_alpha, lr=0.01,
                      corr_bias_scale=corr_bias_scale, n_shared=n_shared,
                      capacity_factor=capacity_factor)


def test_wide_draws_are_within_the_limits():
    for i in WIDE_CASES:
        wl = draw_wide_workload(i)
        assert wl.E <= 256 and 1 <= wl.k <= min(32, wl.E) and wl.n_groups <= 32
        assert wl.D % 8 == 0 and wl.F % 8 == 0
        assert wl.E % wl.n_groups == 0 and wl.k <= wl.topk_groups * (wl.E // wl.n_groups)
        assert wl.dtype == "f32" or wl.E % 8 == 0


@pytest.mark.gpu
@pytest.mark.parametrize("i", WIDE_CASES,
                         ids=[f"wide{i}-E{draw_wide_workload(i).E}-k{draw_wide_workload(i).k}"
                              for i in WIDE_CASES])
def test_wide_random_configuration_step(i):
    errs, _, _ = _one_step_parity(draw_wide_workload(i), seed=5000 + i)
    assert np.isfinite(max(errs.values()))
