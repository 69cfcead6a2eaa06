"""The arithmetic behind the fp32 expert GEMMs on the tensor cores
(csrc/gemm_f32x3.cu), checked on the CPU with torch's bf16 rounding
(round to nearest even, as __float2bfloat16_rn):

* the three bf16 terms of an fp32 value are exact differences and hold the
  value to 2^-24 of its magnitude;
* the reduction over six K blocks laid out as A' = [a3 a2 a1 a2 a1 a1],
  B' = [b1 b2 b3 b1 b2 b1] gives the fp32 operands' dot product to a few
  2^-24 of sum |a b| (the three dropped term products are below 2^-26 of
  |a b| each), far inside the fp32 layers' 1e-4 tolerance, while the plain
  bf16 product (one block) misses it by ~1e-3;
* the block order matters: pairing the terms differently (a mistake in the
  layout tables) breaks that bound.
"""

import numpy as np
import torch

A_TERMS = [2, 1, 0, 1, 0, 0]      # a3 a2 a1 a2 a1 a1: smallest products first
B_TERMS = [0, 1, 2, 0, 1, 0]      # b1 b2 b3 b1 b2 b1


def _terms(x: torch.Tensor):
    t1 = x.to(torch.bfloat16).float()
    r1 = x - t1
    t2 = r1.to(torch.bfloat16).float()
    r2 = r1 - t2
    t3 = r2.to(torch.bfloat16).float()
    return [t1, t2, t3], (r1, r2)


def _expand(x: torch.Tensor, pattern):
    t, _ = _terms(x)
    return torch.cat([t[i] for i in pattern], dim=-1)


def test_terms_are_exact_and_hold_the_value():
    g = torch.Generator().manual_seed(0)
    x = (torch.randn(100000, generator=g) * torch.exp(torch.randn(100000, generator=g) * 4)).float()
    t, (r1, r2) = _terms(x)
    x64 = x.double()
    # the differences are exact in fp32
    assert torch.equal(r1.double(), x64 - t[0].double())
    assert torch.equal(r2.double(), r1.double() - t[1].double())
    err = (x64 - (t[0].double() + t[1].double() + t[2].double())).abs()
    assert torch.all(err <= 2.0 ** -24 * x64.abs())


def test_six_block_reduction_is_fp32_accurate():
    g = torch.Generator().manual_seed(1)
    K, rows = 512, 64
    a = torch.randn(rows, K, generator=g)
    b = torch.randn(rows, K, generator=g)
    exact = (a.double() * b.double()).sum(-1)
    scale = (a.double() * b.double()).abs().sum(-1)
    A = _expand(a, A_TERMS).double()
    B = _expand(b, B_TERMS).double()
    six = (A * B).sum(-1)
    assert torch.all((six - exact).abs() <= 4 * 2.0 ** -24 * scale)
    # one bf16 block alone is three orders of magnitude worse
    one = (a.to(torch.bfloat16).double() * b.to(torch.bfloat16).double()).sum(-1)
    assert np.median(((one - exact).abs() / scale).numpy()) > 1e-4


def test_wrong_pairing_is_detected():
    g = torch.Generator().manual_seed(2)
    a = torch.randn(16, 256, generator=g)
    b = torch.randn(16, 256, generator=g)
    exact = (a.double() * b.double()).sum(-1)
    scale = (a.double() * b.double()).abs().sum(-1)
    # (swapping B's last two blocks would not be a mistake: A's last two
    # blocks are both a1, so the same six products are formed)
    for bad_b in ([0, 1, 2, 0, 1, 1], [0, 1, 2, 0, 2, 0], [0, 2, 2, 0, 1, 0], [1, 1, 2, 0, 1, 0]):
        B = _expand(b, bad_b).double()
        wrong = (_expand(a, A_TERMS).double() * B).sum(-1)
        assert torch.max((wrong - exact).abs() / scale) > 4 * 2.0 ** -24, bad_b
