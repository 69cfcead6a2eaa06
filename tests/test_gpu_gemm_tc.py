"""The tcgen05 grouped GEMM (moe_grouped_gemm) against a plain PyTorch fp32
matmul of the same operands, per expert segment.  Segments include empty
experts, one-row experts and ragged tails; N and K include non-multiples of
the 256 / 64 tile sizes."""

import pytest
import torch

from sparse_mixture_experts_softmax_gb300 import binding as B

pytestmark = pytest.mark.gpu


def _offsets(counts):
    off = [0]
    for c in counts:
        off.append(off[-1] + c)
    return torch.tensor(off, dtype=torch.int32, device="cuda")


def _rel(a, b):
    den = b.abs().max().item()
    return (a - b).abs().max().item() / den if den > 0 else (a - b).abs().max().item()


CASES = [
    ([256], 256, 128),
    ([300, 0, 129, 1, 570], 704, 1024),
    ([128, 256, 0, 0, 77], 256, 64),
    ([5], 512, 200),
    ([1000, 24, 0, 333], 1408, 2048),
    ([5000, 0, 3100, 100, 2600], 704, 1000),
]


@pytest.mark.parametrize("counts,N,K", CASES)
@pytest.mark.parametrize("form", [0, 1])
def test_ragged_m_forms(form, counts, N, K):
    g = torch.Generator(device="cuda")
    g.manual_seed(1)
    E, M = len(counts), sum(counts)
    off = _offsets(counts)
    A = torch.randn(M, K, generator=g, device="cuda").to(torch.bfloat16)
    Bw = (torch.randn(E, N, K, generator=g, device="cuda") / K ** 0.5).to(torch.bfloat16)
    Bt = Bw if form == 0 else Bw.transpose(1, 2).contiguous()     # [E, K, N] for form 1
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_grouped_gemm(form, M, N, K, E, off, A, Bt, C, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    o = off.tolist()
    for e in range(E):
        if counts[e] == 0:
            continue
        ref = A[o[e]:o[e + 1]].float() @ Bw[e].float().T
        got = C[o[e]:o[e + 1]].float()
        assert torch.isfinite(got).all(), e
        assert _rel(got, ref) <= 1e-2, (e, _rel(got, ref))


@pytest.mark.parametrize("counts,Mo,N", [([300, 0, 129, 1, 570], 1024, 704),
                                         ([64, 65, 0, 127], 704, 256),
                                         ([2000, 3], 512, 2048),
                                         # skewed loads: the largest expert holds more than
                                         # twice the mean rows (the case a MOE_TC_SNAKE
                                         # build deals in size order), empty experts
                                         ([4000, 0, 10, 3000, 0, 1, 64, 65, 128, 500], 512, 768)])
def test_ragged_k_form(counts, Mo, N):
    g = torch.Generator(device="cuda")
    g.manual_seed(2)
    E, R = len(counts), sum(counts)
    off = _offsets(counts)
    A = torch.randn(R, Mo, generator=g, device="cuda").to(torch.bfloat16)
    Bm = torch.randn(R, N, generator=g, device="cuda").to(torch.bfloat16)
    C = torch.full((E, Mo, N), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_grouped_gemm(2, Mo, N, R, E, off, A, Bm, C, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    o = off.tolist()
    for e in range(E):
        ref = A[o[e]:o[e + 1]].float().T @ Bm[o[e]:o[e + 1]].float()
        if counts[e] == 0:
            assert torch.equal(C[e], torch.zeros_like(C[e])), e
        else:
            assert _rel(C[e], ref) <= 1e-4, (e, _rel(C[e], ref))


def test_repeatable_bits():
    counts, N, K = [200, 0, 313], 512, 512
    E, M = len(counts), sum(counts)
    off = _offsets(counts)
    A = torch.randn(M, K, device="cuda").to(torch.bfloat16)
    Bw = torch.randn(E, N, K, device="cuda").to(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    C1 = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    C2 = torch.empty_like(C1)
    B.moe_grouped_gemm(0, M, N, K, E, off, A, Bw, C1, st)
    B.moe_grouped_gemm(0, M, N, K, E, off, A, Bw, C2, st)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)


def test_bounded_wait_times_out_and_context_survives():
    """Failure detection without a fault: with every load withheld the kernel's
    bounded waits expire, it stops cleanly and reports MOE_ERR_TIMEOUT in the
    device status word; the same context then runs a normal GEMM correctly."""
    counts, N, K = [300, 0, 129], 512, 256
    E, M = len(counts), sum(counts)
    off = _offsets(counts)
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    A = torch.randn(M, K, generator=g, device="cuda").to(torch.bfloat16)
    Bw = (torch.randn(E, N, K, generator=g, device="cuda") / K ** 0.5).to(torch.bfloat16)
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_selftest_wait_timeout(0, M, N, K, E, off, A, Bw, C, st, 20_000_000)   # 20 ms
    torch.cuda.synchronize()
    assert st.item() == 6                        # MOE_ERR_TIMEOUT
    assert torch.isnan(C.float()).all()          # nothing was stored
    st.zero_()
    B.moe_grouped_gemm(0, M, N, K, E, off, A, Bw, C, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    o = off.tolist()
    for e in range(E):
        if counts[e]:
            ref = A[o[e]:o[e + 1]].float() @ Bw[e].float().T
            assert _rel(C[o[e]:o[e + 1]].float(), ref) <= 1e-2


@pytest.mark.parametrize("form,raw", [(0, [0, 100, 50, 400]), (0, [0, 100, 50, 220]),
                                      (1, [-7, 64, 64, 1000]), (2, [0, 900, 20, 20])])
def test_caller_offsets_are_clamped(form, raw):
    """Offsets from a caller that run past the total rows, go negative or
    decrease are clamped on the device to a non-decreasing sequence within
    [0, total rows]: the result equals the GEMM over the clamped segments and
    nothing past the end of C is written (a guard region behind C keeps its
    sentinel)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(4)
    E = len(raw) - 1
    rows = 300
    clamped, prev = [], 0
    for v in raw:
        prev = min(max(v, prev), rows)
        clamped.append(prev)
    off = torch.tensor(raw, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    guard = 4096
    if form in (0, 1):
        N, K = 256, 128
        A = torch.randn(rows, K, generator=g, device="cuda").to(torch.bfloat16)
        Bw = (torch.randn(E, N, K, generator=g, device="cuda") / K ** 0.5).to(torch.bfloat16)
        Bt = Bw if form == 0 else Bw.transpose(1, 2).contiguous()
        buf = torch.full((rows * N + guard,), 7.0, dtype=torch.bfloat16, device="cuda")
        C = buf[: rows * N].view(rows, N)
        B.moe_grouped_gemm(form, rows, N, K, E, off, A, Bt, C, st)
        torch.cuda.synchronize()
        for e in range(E):
            lo, hi = clamped[e], clamped[e + 1]
            if hi > lo:
                ref = A[lo:hi].float() @ Bw[e].float().T
                assert _rel(C[lo:hi].float(), ref) <= 1e-2, e
        # rows outside every clamped segment are not written
        assert torch.all(C[clamped[-1]:] == 7.0)
        assert torch.all(buf[rows * N:] == 7.0)
    else:
        Mo, N = 128, 256
        A = torch.randn(rows, Mo, generator=g, device="cuda").to(torch.bfloat16)
        Bm = torch.randn(rows, N, generator=g, device="cuda").to(torch.bfloat16)
        buf = torch.full((E * Mo * N + guard,), 7.0, dtype=torch.float32, device="cuda")
        C = buf[: E * Mo * N].view(E, Mo, N)
        B.moe_grouped_gemm(2, Mo, N, rows, E, off, A, Bm, C, st)
        torch.cuda.synchronize()
        for e in range(E):
            lo, hi = clamped[e], clamped[e + 1]
            ref = A[lo:hi].float().T @ Bm[lo:hi].float()
            if hi == lo:
                assert torch.equal(C[e], torch.zeros_like(C[e])), e
            else:
                assert _rel(C[e], ref) <= 1e-4, e
        assert torch.all(buf[E * Mo * N:] == 7.0)
    assert st.item() == 0

