"""The C ABI library loads, exports every entry point include/moe.h declares,
and rejects bad arguments on the host (no GPU needed: validation runs before
any CUDA call)."""

import ctypes
import os
import re

import pytest

from sparse_mixture_experts_softmax_gb300 import binding as B
from sparse_mixture_experts_softmax_gb300.build import INCLUDE, LIB, build_library


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(LIB):
        build_library()
    return B.lib()


def _declared():
    names = []
    for f in os.listdir(INCLUDE):
        if f.endswith(".h"):
            txt = open(os.path.join(INCLUDE, f)).read()
            names += re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", txt)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n


def _cfg(**kw):
    base = dict(T=64, D=32, F=64, E=4, k=2, act="relu", score="softmax", dtype="f32",
                has_bias=True, aux_alpha=0.01)
    base.update(kw)
    return B.make_config(**base)


def test_workspace_size_valid_and_invalid(L):
    assert B.moe_workspace_size(_cfg()) > 0
    assert B.moe_workspace_size(_cfg(T=0)) > 0
    assert B.moe_workspace_size(_cfg(k=0)) == 0
    assert B.moe_workspace_size(_cfg(k=5)) == 0                 # k > E
    assert B.moe_workspace_size(_cfg(E=300, k=2)) == 0          # E > 256
    assert B.moe_workspace_size(_cfg(D=30)) == 0                # D % 8
    assert B.moe_workspace_size(_cfg(act="swiglu", has_bias=True)) == 0
    assert B.moe_workspace_size(_cfg(E=8, n_groups=3, topk_groups=1)) == 0
    assert B.moe_workspace_size(_cfg(E=8, k=4, n_groups=4, topk_groups=1)) == 0  # k > kept
    # shared experts: SwiGLU and bf16 only
    assert B.moe_workspace_size(_cfg(n_shared=1)) == 0
    assert B.moe_workspace_size(_cfg(E=8, act="swiglu", has_bias=False, dtype="bf16",
                                     n_shared=2)) > \
        B.moe_workspace_size(_cfg(E=8, act="swiglu", has_bias=False, dtype="bf16"))
    assert B.moe_workspace_size(_cfg(n_shared=-1)) == 0
    assert B.moe_host_staging_size(_cfg()) >= 64 * 32 * 8


def test_workspace_grows_with_tokens(L):
    a = B.moe_workspace_size(_cfg(T=64))
    b = B.moe_workspace_size(_cfg(T=6400))
    assert b > a


class _Fake:
    """Stands in for a tensor: a fake, aligned address (never dereferenced)."""
    def __init__(self, addr, n=1 << 40):
        self.addr, self.n = addr, n

    def is_contiguous(self):
        return True

    def data_ptr(self):
        return self.addr

    def numel(self):
        return self.n


def _status(fn, *a):
    with pytest.raises(B.MoEError) as ei:
        fn(*a)
    return ei.value.status


def test_host_validation_errors(L):
    good = lambda i: _Fake(0x10000 * (i + 1))  # noqa: E731
    w = B.make_weights(good(1), good(2), good(3), b1=good(4), b2=good(5))
    ws = _Fake(0x900000, 1 << 40)
    assert _status(B.moe_forward, _cfg(k=0), w, good(6), good(7), ws) == B.MOE_ERR_INVALID_ARG
    assert _status(B.moe_forward, _cfg(E=512, k=2), w, good(6), good(7), ws) == B.MOE_ERR_UNSUPPORTED
    # missing bias pointers for a biased layer
    w_nob = B.make_weights(good(1), good(2), good(3))
    assert _status(B.moe_forward, _cfg(), w_nob, good(6), good(7), ws) == B.MOE_ERR_INVALID_ARG
    # misaligned weight / input
    w_bad = B.make_weights(_Fake(0x10008), good(2), good(3), b1=good(4), b2=good(5))
    assert _status(B.moe_forward, _cfg(), w_bad, good(6), good(7), ws) == B.MOE_ERR_ALIGNMENT
    assert _status(B.moe_forward, _cfg(), w, _Fake(0x60004), good(7), ws) == B.MOE_ERR_ALIGNMENT
    # workspace too small
    small = _Fake(0x900000, 1024)
    assert _status(B.moe_forward, _cfg(), w, good(6), good(7), small) == B.MOE_ERR_WORKSPACE_TOO_SMALL
    # SwiGLU needs W3
    cs = _cfg(act="swiglu", has_bias=False)
    w_no3 = B.make_weights(good(1), good(2), good(3))
    assert _status(B.moe_forward, cs, w_no3, good(6), good(7), ws) == B.MOE_ERR_INVALID_ARG
    # backward: grads required
    g_missing = B.make_grads(good(8), good(9), None)
    assert _status(B.moe_backward, _cfg(), w, good(6), good(7), g_missing, None, ws) == B.MOE_ERR_INVALID_ARG
    # train step: bf16 layer without bf16 copies
    g = B.make_grads(good(8), good(9), good(10), db1=good(11), db2=good(12))
    p = B.make_params(good(1), good(2), good(3), g, b1=good(4), b2=good(5))
    assert _status(B.moe_train_step, _cfg(dtype="bf16", E=8), p, good(6), good(7), 0.1, good(13), ws) \
        == B.MOE_ERR_INVALID_ARG
    # bf16 layers need E % 8 == 0 (16-byte rows of the bf16 router operands)
    assert _status(B.moe_train_step, _cfg(dtype="bf16", E=4), p, good(6), good(7), 0.1, good(13), ws) \
        == B.MOE_ERR_UNSUPPORTED
    # train step: gradient buffers are optional, but those given must be aligned
    g_odd = B.make_grads(good(8), _Fake(0x90004), None, db1=good(11), db2=good(12))
    p_odd = B.make_params(good(1), good(2), good(3), g_odd, b1=good(4), b2=good(5))
    assert _status(B.moe_train_step, _cfg(), p_odd, good(6), good(7), 0.1, good(13), ws) \
        == B.MOE_ERR_ALIGNMENT


def test_selftest_rejects_unbounded_wait_limit(L):
    good = lambda i: _Fake(0x10000 * (i + 1))  # noqa: E731
    for bad in (0, -1, 3_000_000_000):
        assert _status(B.moe_selftest_wait_timeout, 0, 1, 8, 8, 1, good(1), good(2), good(3),
                       good(4), good(5), bad) == B.MOE_ERR_INVALID_ARG


def test_pipelined_host_steps_validation(L):
    good = lambda i: _Fake(0x10000 * (i + 1))  # noqa: E731
    g = B.make_grads(good(8), good(9), good(10), db1=good(11), db2=good(12))
    p = B.make_params(good(1), good(2), good(3), g, b1=good(4), b2=good(5))
    ws = _Fake(0x900000, 1 << 40)
    small = _Fake(0xA00000, B.moe_host_staging_size(_cfg()))   # one slot, two needed
    assert _status(B.moe_train_steps_host, _cfg(), p, [good(6)], [good(7)], 0.1, good(13),
                   small, ws) == B.MOE_ERR_WORKSPACE_TOO_SMALL
    assert _status(B.moe_train_steps_host, _cfg(), p, [good(6)], [good(7)], 0.1, good(13),
                   _Fake(0xA00008, 1 << 30), ws) == B.MOE_ERR_ALIGNMENT


def test_inspection_accessors_validation(L):
    good = lambda i: _Fake(0x10000 * (i + 1))  # noqa: E731
    ws = _Fake(0x900000, 1 << 40)
    small = _Fake(0x900000, 1024)
    # workspace checks before any copy
    assert _status(B.moe_get_hidden, _cfg(), small, good(1)) == B.MOE_ERR_WORKSPACE_TOO_SMALL
    assert _status(B.moe_get_hidden, _cfg(), _Fake(0x900008, 1 << 40), good(1)) \
        == B.MOE_ERR_ALIGNMENT
    assert _status(B.moe_get_intermediates, _cfg(), small, good(1)) \
        == B.MOE_ERR_WORKSPACE_TOO_SMALL
    # H3 exists only for SwiGLU experts
    assert _status(B.moe_get_hidden, _cfg(), ws, good(1), good(2)) == B.MOE_ERR_INVALID_ARG
    # an invalid configuration is refused first
    assert _status(B.moe_get_hidden, _cfg(k=0), ws, good(1)) == B.MOE_ERR_INVALID_ARG


def test_status_strings(L):
    for s in range(7):
        assert B.moe_status_string(s)
    assert "workspace" in B.moe_status_string(B.MOE_ERR_WORKSPACE_TOO_SMALL)


def test_expert_parallel_validation(L):
    """The expert-parallel phases check their requests on the host."""
    cfg = _cfg(E=8, act="swiglu", has_bias=False, dtype="bf16")
    assert B.moe_ep_workspace_size(cfg, B.moe_ep_config(2, 0, 128)) > 0
    assert B.moe_ep_workspace_size(cfg, B.moe_ep_config(3, 0, 128)) == 0   # 3 does not divide E
    assert B.moe_ep_workspace_size(cfg, B.moe_ep_config(2, 2, 128)) == 0   # rank out of range
    assert B.moe_ep_workspace_size(cfg, B.moe_ep_config(2, 0, 10)) == 0    # T_total < T
    cap = _cfg(E=8, act="swiglu", has_bias=False, dtype="bf16", capacity_factor=1.0)
    assert B.moe_ep_workspace_size(cap, B.moe_ep_config(2, 0, 128)) == 0   # no capacity here
    # the source-side workspace holds no expert-MLP buffers
    assert B.moe_ep_workspace_size(cfg, B.moe_ep_config(2, 0, 128)) < B.moe_workspace_size(cfg)
    offs = B.moe_ep_buffer_offsets(cfg, B.moe_ep_config(2, 1, 128))
    assert offs == sorted(offs) and offs[0] % 256 == 0
    good = lambda i: _Fake(0x10000 * (i + 1))  # noqa: E731
    ws = _Fake(0x900000, 1 << 40)
    ep = B.moe_ep_config(2, 0, 128)
    w = B.make_weights(good(1), None, None)
    assert _status(B.moe_ep_route, cfg, ep, w, good(2), None, ws) == B.MOE_ERR_INVALID_ARG
    assert _status(B.moe_ep_route, cfg, ep, w, good(2), _Fake(0x30004), ws) == B.MOE_ERR_ALIGNMENT
    small = _Fake(0x900000, 1024)
    assert _status(B.moe_ep_route, cfg, ep, w, good(2), good(3), small) \
        == B.MOE_ERR_WORKSPACE_TOO_SMALL
    # received rows beyond what every rank could route are refused
    rows = B.make_ep_rows(128 * 2 + 1, good(4), good(5), good(6), good(7), good(8), good(9),
                          status=good(10))
    wx = B.make_weights(None, good(1), good(2), good(3))
    assert _status(B.moe_ep_expert_forward, cfg, ep, wx, rows) == B.MOE_ERR_INVALID_ARG


def test_debug_variant_and_poke_refusal(L):
    """The release library reports no debug checks and refuses the fault
    injection entry point before touching the device; the MOE_DEBUG variant
    (built beside it) exports the same symbols and reports its checks."""
    assert B.moe_build_flags() == 0
    ws = _Fake(0x900000, 1 << 40)
    assert _status(B.moe_debug_poke_routing, _cfg(), ws, 1, 0, 5) == B.MOE_ERR_UNSUPPORTED
    from sparse_mixture_experts_softmax_gb300.build import LIB_DEBUG
    if not os.path.exists(LIB_DEBUG):
        build_library(debug=True)
    dbg = ctypes.CDLL(LIB_DEBUG)
    for n in _declared():
        assert hasattr(dbg, n), n
    with B.use_library(debug=True):
        assert B.moe_build_flags() == B.MOE_BUILD_DEBUG_CHECKS
        # host-side validation of the injection itself, before any device work
        assert _status(B.moe_debug_poke_routing, _cfg(), ws, 2, 0, 5) == B.MOE_ERR_INVALID_ARG
        assert _status(B.moe_debug_poke_routing, _cfg(), ws, 1, 64 * 2, 5) == B.MOE_ERR_INVALID_ARG


def test_expert_gemm_path(L):
    """Which units run a layer's expert GEMMs: bf16 layers the tensor cores;
    fp32 layers with D F >= 65536 the tensor cores through the three-term
    bf16 split while its scratch (12 bytes per expanded fp32 value, the
    largest operand pair of the layer) stays within 1 GiB, else the CUDA
    cores; the scratch is part of the workspace exactly when that path is
    taken."""
    bf = _cfg(dtype="bf16", D=64, F=64, E=8, has_bias=False, act="swiglu")
    assert B.moe_expert_gemm_path(bf) == B.GEMM_TENSOR_BF16
    assert B.moe_expert_gemm_path(_cfg()) == B.GEMM_CUDA_CORES        # D F = 2048: too small
    assert B.moe_expert_gemm_path(_cfg(D=256, F=256)) == B.GEMM_TENSOR_F32X3
    # R = 65536 rows of D = F = 1024 over 64 experts: 805 MB + 805 MB of operands
    big = _cfg(T=8192, k=8, E=64, D=1024, F=1024)
    assert B.moe_expert_gemm_path(big) == B.GEMM_CUDA_CORES
    assert B.moe_expert_gemm_path(_cfg(k=0)) < 0
    # dense fp32 layer of the benchmarks: R = 8192, D = 512, F = 1024, E = 8
    dense = _cfg(T=4096, k=2, E=8, D=512, F=1024, act="gelu_tanh")
    assert B.moe_expert_gemm_path(dense) == B.GEMM_TENSOR_F32X3
    R, D, F, E = 8192, 512, 1024, 8
    want = 12 * (R * F + E * D * F)          # down / dXe: the largest pair
    assert B.moe_workspace_size(dense) > want
    # expert-parallel ranks size their own scratch by the rows they received
    ep = B.moe_ep_config(2, 0, 4096)
    r, el = 4096, E // 2
    assert B.moe_ep_f32_scratch_size(dense, ep, r) == max(
        12 * (r * D + el * F * D), 12 * (r * F + el * D * F),
        12 * (r * D + r * F) + 256)     # dW: six blocks of rows of both operands, scaled offsets
    assert B.moe_ep_f32_scratch_size(dense, ep, 4096 * 2 + 1) == 0     # more than T_total k rows
    assert B.moe_ep_f32_scratch_size(bf, B.moe_ep_config(2, 0, 64), 8) == 0
