"""ctypes binding of ``libmoe_gb300.so`` (the C ABI declared in ``include/moe.h``).

Argument marshalling only: every function here forwards torch tensors' device
pointers and sizes to the entry point of the same name, and raises
``MoEError`` when the library returns a status other than ``MOE_OK``.  No step
of the layer is computed in Python, and there is no fallback: if the library
is missing, every call raises.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe_gb300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_ALIGNMENT = 3
MOE_ERR_WORKSPACE_TOO_SMALL = 4
MOE_ERR_CUDA = 5
MOE_ERR_TIMEOUT = 6
MOE_BUILD_DEBUG_CHECKS = 1

ACT = {"relu": 0, "gelu_tanh": 1, "swiglu": 2}
SCORE = {"softmax": 0, "sigmoid": 1}
GROUP_SCORE = {"top2_sum": 0, "max": 1}
DTYPE = {"f32": 0, "bf16": 1}

c_int32, c_float, c_void_p, c_size_t = ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t


class moe_config(ctypes.Structure):
    _fields_ = [("T", c_int32), ("D", c_int32), ("F", c_int32), ("E", c_int32), ("k", c_int32),
                ("n_groups", c_int32), ("topk_groups", c_int32), ("group_score", c_int32),
                ("act", c_int32), ("score", c_int32), ("dtype", c_int32), ("has_bias", c_int32),
                ("aux_alpha", c_float), ("n_shared", c_int32), ("capacity_factor", c_float)]


class moe_weights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("w_gate", "w1", "w3", "w2", "b1", "b2", "logit_bias",
                                        "corr_bias", "ws1", "ws3", "ws2")]


class moe_grads(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("dw_gate", "dw1", "dw3", "dw2", "db1", "db2",
                                        "dws1", "dws3", "dws2")]


class moe_params(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("w_gate", "w1", "w3", "w2", "b1", "b2",
                                        "w1_lp", "w3_lp", "w2_lp", "logit_bias", "corr_bias",
                                        "ws1", "ws3", "ws2", "ws1_lp", "ws3_lp", "ws2_lp")] + \
               [("grads", moe_grads)]


class moe_ep_config(ctypes.Structure):
    _fields_ = [("n_ranks", c_int32), ("rank", c_int32), ("T_total", c_int32)]


class moe_ep_rows(ctypes.Structure):
    _fields_ = [("rows", c_int32)] + [(n, c_void_p) for n in (
        "offsets", "x", "h1", "h3", "a", "y", "dy", "dh1", "dh3", "dx", "status",
        "f32_scratch")] + [("f32_scratch_bytes", ctypes.c_size_t)]


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn}: {text} (status {status})")
        self.status = status


_LIB_DEBUG_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                               "libmoe_gb300_debug.so")
_lib = None          # the library every call below goes through
_loaded = {}         # path -> loaded handle


def lib() -> ctypes.CDLL:
    """The loaded library (the release build unless ``use_library`` switched
    to the MOE_DEBUG variant); raises if it has not been built."""
    global _lib
    if _lib is None:
        _lib = _load(_LIB_PATH)
    return _lib


class use_library:
    """``with use_library(debug=True): ...`` routes every call of this module
    to the MOE_DEBUG variant (device-side index checks) for the block."""

    def __init__(self, debug: bool):
        self.path = _LIB_DEBUG_PATH if debug else _LIB_PATH

    def __enter__(self):
        global _lib
        self.saved = _lib
        _lib = _load(self.path)
        return _lib

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def _load(path: str) -> ctypes.CDLL:
    if path in _loaded:
        return _loaded[path]
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "sparse_mixture_experts_softmax_gb300.build.build_library()")
    L = ctypes.CDLL(path)
    P = ctypes.POINTER
    L.moe_workspace_size.argtypes = [P(moe_config)]
    L.moe_workspace_size.restype = c_size_t
    L.moe_host_staging_size.argtypes = [P(moe_config)]
    L.moe_host_staging_size.restype = c_size_t
    L.moe_forward.argtypes = [P(moe_config), P(moe_weights), c_void_p, c_void_p, c_void_p,
                              c_size_t, c_void_p]
    L.moe_backward.argtypes = [P(moe_config), P(moe_weights), c_void_p, c_void_p, P(moe_grads),
                               c_void_p, c_void_p, c_size_t, c_void_p]
    L.moe_train_step.argtypes = [P(moe_config), P(moe_params), c_void_p, c_void_p, c_float,
                                 c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]
    L.moe_train_step_host.argtypes = [P(moe_config), P(moe_params), c_void_p, c_void_p,
                                      c_float, c_void_p, c_void_p, c_size_t, c_void_p,
                                      c_size_t, c_void_p]
    L.moe_train_steps_host.argtypes = [P(moe_config), P(moe_params), c_int32, c_void_p,
                                       c_void_p, c_float, c_void_p, c_void_p, c_size_t,
                                       c_void_p, c_size_t, c_void_p]
    L.moe_get_routing.argtypes = [P(moe_config), c_void_p, c_size_t] + [c_void_p] * 8
    L.moe_get_intermediates.argtypes = [P(moe_config), c_void_p, c_size_t, c_void_p, c_void_p,
                                        c_void_p, c_void_p]
    L.moe_status_string.argtypes = [c_int32]
    L.moe_status_string.restype = ctypes.c_char_p
    L.moe_last_launch_count.argtypes = []
    L.moe_last_launch_count.restype = c_int32
    L.moe_profile_enable.argtypes = [c_int32]
    L.moe_profile_enable.restype = None
    L.moe_profile_count.argtypes = []
    L.moe_profile_count.restype = c_int32
    L.moe_profile_name.argtypes = [c_int32]
    L.moe_profile_name.restype = ctypes.c_char_p
    L.moe_profile_ms.argtypes = [c_int32]
    L.moe_profile_ms.restype = c_float
    L.moe_dispatch_noalloc.argtypes = [P(moe_config)] + [c_void_p] * 6
    L.moe_device_status.argtypes = [P(moe_config), c_void_p, c_size_t, c_void_p, c_void_p]
    L.moe_get_hidden.argtypes = [P(moe_config), c_void_p, c_size_t, c_void_p, c_void_p,
                                 c_void_p]
    L.moe_grouped_gemm.argtypes = [c_int32] * 5 + [c_void_p] * 6
    L.moe_selftest_wait_timeout.argtypes = [c_int32] * 5 + [c_void_p] * 5 + [ctypes.c_int64,
                                                                            c_void_p]
    L.moe_ep_workspace_size.argtypes = [P(moe_config), P(moe_ep_config)]
    L.moe_ep_workspace_size.restype = c_size_t
    L.moe_ep_f32_scratch_size.argtypes = [P(moe_config), P(moe_ep_config), c_int32]
    L.moe_ep_f32_scratch_size.restype = c_size_t
    L.moe_ep_buffer_offsets.argtypes = [P(moe_config), P(moe_ep_config), P(c_size_t)]
    L.moe_ep_route.argtypes = [P(moe_config), P(moe_ep_config), P(moe_weights), c_void_p,
                               c_void_p, c_void_p, c_size_t, c_void_p]
    L.moe_ep_expert_forward.argtypes = [P(moe_config), P(moe_ep_config), P(moe_weights),
                                        P(moe_ep_rows), c_void_p]
    L.moe_ep_combine.argtypes = [P(moe_config), P(moe_ep_config), c_void_p, c_void_p,
                                 c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]
    L.moe_ep_expert_backward.argtypes = [P(moe_config), P(moe_ep_config), P(moe_params),
                                         P(moe_ep_rows), c_float, c_void_p]
    L.moe_ep_router_backward.argtypes = [P(moe_config), P(moe_ep_config), c_void_p, c_void_p,
                                         c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]
    L.moe_ep_router_update.argtypes = [P(moe_config), c_void_p, c_void_p, c_float, c_void_p]
    L.moe_ep_get_routing.argtypes = [P(moe_config), P(moe_ep_config), c_void_p, c_size_t] + \
        [c_void_p] * 8
    for fn in ("moe_ep_buffer_offsets", "moe_ep_get_routing", "moe_ep_route",
               "moe_ep_expert_forward",
               "moe_ep_combine", "moe_ep_expert_backward", "moe_ep_router_backward",
               "moe_ep_router_update"):
        getattr(L, fn).restype = c_int32
    for fn in ("moe_forward", "moe_backward", "moe_train_step", "moe_train_step_host",
               "moe_train_steps_host",
               "moe_get_routing", "moe_get_intermediates", "moe_get_hidden",
               "moe_dispatch_noalloc",
               "moe_device_status", "moe_grouped_gemm", "moe_selftest_wait_timeout"):
        getattr(L, fn).restype = c_int32
    L.moe_build_flags.argtypes = []
    L.moe_build_flags.restype = c_int32
    L.moe_expert_gemm_path.argtypes = [P(moe_config)]
    L.moe_expert_gemm_path.restype = c_int32
    L.moe_debug_poke_routing.argtypes = [P(moe_config), c_void_p, c_size_t, c_int32,
                                         ctypes.c_int64, c_int32, c_void_p]
    L.moe_debug_poke_routing.restype = c_int32
    _loaded[path] = L
    return L


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the MoE library must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        if torch.cuda.is_available():
            return torch.cuda.current_stream().cuda_stream
        return None
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(fn: str, status: int):
    if status != MOE_OK:
        raise MoEError(fn, status, lib().moe_status_string(status).decode())


def make_config(T, D, F, E, k, act="relu", score="softmax", n_groups=1, topk_groups=1,
                group_score="top2_sum", dtype="f32", has_bias=True, aux_alpha=0.0,
                n_shared=0, capacity_factor=0.0) -> moe_config:
    return moe_config(T, D, F, E, k, n_groups, topk_groups, GROUP_SCORE[group_score], ACT[act],
                      SCORE[score], DTYPE[dtype], int(bool(has_bias)), float(aux_alpha),
                      int(n_shared), float(capacity_factor))


def make_weights(w_gate, w1, w2, w3=None, b1=None, b2=None, logit_bias=None,
                 corr_bias=None, ws1=None, ws3=None, ws2=None) -> moe_weights:
    return moe_weights(_ptr(w_gate), _ptr(w1), _ptr(w3), _ptr(w2), _ptr(b1), _ptr(b2),
                       _ptr(logit_bias), _ptr(corr_bias), _ptr(ws1), _ptr(ws3), _ptr(ws2))


def make_grads(dw_gate, dw1, dw2, dw3=None, db1=None, db2=None, dws1=None, dws3=None,
               dws2=None) -> moe_grads:
    return moe_grads(_ptr(dw_gate), _ptr(dw1), _ptr(dw3), _ptr(dw2), _ptr(db1), _ptr(db2),
                     _ptr(dws1), _ptr(dws3), _ptr(dws2))


def make_params(w_gate, w1, w2, grads: moe_grads, w3=None, b1=None, b2=None, w1_lp=None,
                w3_lp=None, w2_lp=None, logit_bias=None, corr_bias=None, ws1=None, ws3=None,
                ws2=None, ws1_lp=None, ws3_lp=None, ws2_lp=None) -> moe_params:
    return moe_params(_ptr(w_gate), _ptr(w1), _ptr(w3), _ptr(w2), _ptr(b1), _ptr(b2),
                      _ptr(w1_lp), _ptr(w3_lp), _ptr(w2_lp), _ptr(logit_bias), _ptr(corr_bias),
                      _ptr(ws1), _ptr(ws3), _ptr(ws2), _ptr(ws1_lp), _ptr(ws3_lp), _ptr(ws2_lp),
                      grads)


def moe_workspace_size(cfg: moe_config) -> int:
    return int(lib().moe_workspace_size(ctypes.byref(cfg)))


def moe_host_staging_size(cfg: moe_config) -> int:
    return int(lib().moe_host_staging_size(ctypes.byref(cfg)))


def moe_forward(cfg, weights, x, y, workspace, stream=None):
    _check("moe_forward", lib().moe_forward(ctypes.byref(cfg), ctypes.byref(weights), _ptr(x),
                                            _ptr(y), _ptr(workspace), workspace.numel(),
                                            _stream(stream)))


def moe_backward(cfg, weights, x, dy, grads, dx, workspace, stream=None):
    _check("moe_backward", lib().moe_backward(ctypes.byref(cfg), ctypes.byref(weights), _ptr(x),
                                              _ptr(dy), ctypes.byref(grads), _ptr(dx),
                                              _ptr(workspace), workspace.numel(), _stream(stream)))


def moe_train_step(cfg, params, x, y_target, lr, d_loss, workspace, dx=None, stream=None):
    _check("moe_train_step", lib().moe_train_step(ctypes.byref(cfg), ctypes.byref(params), _ptr(x),
                                                  _ptr(y_target), float(lr), _ptr(d_loss),
                                                  _ptr(dx), _ptr(workspace), workspace.numel(),
                                                  _stream(stream)))


def moe_train_step_host(cfg, params, x_host, y_target_host, lr, loss_host, staging, workspace,
                        stream=None):
    """x_host / y_target_host / loss_host are CPU tensors (pinned for full speed)."""
    _check("moe_train_step_host",
           lib().moe_train_step_host(ctypes.byref(cfg), ctypes.byref(params), _ptr(x_host),
                                     _ptr(y_target_host), float(lr), _ptr(loss_host),
                                     _ptr(staging), staging.numel(), _ptr(workspace),
                                     workspace.numel(), _stream(stream)))


def moe_train_steps_host(cfg, params, x_hosts, y_target_hosts, lr, loss_host, staging, workspace,
                         stream=None):
    """Pipelined steps over host batches (lists of CPU tensors, pinned for full
    speed); loss_host is a CPU float32 tensor of 2 * len(x_hosts) values and
    staging a device buffer of 2 * moe_host_staging_size(cfg) bytes."""
    n = len(x_hosts)
    if len(y_target_hosts) != n:
        raise ValueError("one target batch per input batch")
    xs = (c_void_p * max(n, 1))(*[_ptr(t) for t in x_hosts])
    ts = (c_void_p * max(n, 1))(*[_ptr(t) for t in y_target_hosts])
    _check("moe_train_steps_host",
           lib().moe_train_steps_host(ctypes.byref(cfg), ctypes.byref(params), int(n), xs, ts,
                                      float(lr), _ptr(loss_host), _ptr(staging), staging.numel(),
                                      _ptr(workspace), workspace.numel(), _stream(stream)))


def moe_get_routing(cfg, workspace, scores=None, idx=None, gate=None, counts=None, offsets=None,
                    src_tok=None, slot_of=None, stream=None):
    _check("moe_get_routing",
           lib().moe_get_routing(ctypes.byref(cfg), _ptr(workspace), workspace.numel(),
                                 _ptr(scores), _ptr(idx), _ptr(gate), _ptr(counts), _ptr(offsets),
                                 _ptr(src_tok), _ptr(slot_of), _stream(stream)))


def moe_get_intermediates(cfg, workspace, ye=None, dxe=None, dlogits=None, stream=None):
    _check("moe_get_intermediates",
           lib().moe_get_intermediates(ctypes.byref(cfg), _ptr(workspace), workspace.numel(),
                                       _ptr(ye), _ptr(dxe), _ptr(dlogits), _stream(stream)))


def moe_get_hidden(cfg, workspace, h1=None, h3=None, stream=None):
    _check("moe_get_hidden",
           lib().moe_get_hidden(ctypes.byref(cfg), _ptr(workspace), workspace.numel(),
                                _ptr(h1), _ptr(h3), _stream(stream)))


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def moe_last_launch_count() -> int:
    return int(lib().moe_last_launch_count())


def moe_profile_enable(on: bool):
    lib().moe_profile_enable(1 if on else 0)


def moe_profile_read():
    """[(kernel name, milliseconds)] of the last call on this thread (waits)."""
    L = lib()
    return [(L.moe_profile_name(i).decode(), float(L.moe_profile_ms(i)))
            for i in range(L.moe_profile_count())]


MOE_NOALLOC_MAX_ROUTED = 1024 * 1024


def moe_dispatch_noalloc(cfg, idx, counts, offsets, src_tok, slot_of, stream=None):
    """Dispatch with the library's fixed scratch array (no allocation, no
    workspace); see include/moe.h."""
    _check("moe_dispatch_noalloc",
           lib().moe_dispatch_noalloc(ctypes.byref(cfg), _ptr(idx), _ptr(counts), _ptr(offsets),
                                      _ptr(src_tok), _ptr(slot_of), _stream(stream)))


def moe_device_status(cfg, workspace, stream=None) -> int:
    out = ctypes.c_int32(0)
    _check("moe_device_status",
           lib().moe_device_status(ctypes.byref(cfg), _ptr(workspace), workspace.numel(),
                                   ctypes.addressof(out), _stream(stream)))
    return int(out.value)


def moe_grouped_gemm(form, M, N, K, E, offsets, A, B, C, dev_status, stream=None):
    """Grouped bf16 GEMM on the tensor cores (see include/moe.h)."""
    _check("moe_grouped_gemm",
           lib().moe_grouped_gemm(int(form), int(M), int(N), int(K), int(E), _ptr(offsets),
                                  _ptr(A), _ptr(B), _ptr(C), _ptr(dev_status), _stream(stream)))


def moe_selftest_wait_timeout(form, M, N, K, E, offsets, A, B, C, dev_status, limit_ns,
                              stream=None):
    """The grouped GEMM with its loads withheld: its bounded waits must expire."""
    _check("moe_selftest_wait_timeout",
           lib().moe_selftest_wait_timeout(int(form), int(M), int(N), int(K), int(E),
                                           _ptr(offsets), _ptr(A), _ptr(B), _ptr(C),
                                           _ptr(dev_status), int(limit_ns), _stream(stream)))


# ---- expert-parallel phases (include/moe_ep.h)

def make_ep_rows(rows: int, offsets, x=None, h1=None, h3=None, a=None, y=None, dy=None,
                 dh1=None, dh3=None, dx=None, status=None, f32_scratch=None) -> moe_ep_rows:
    nbytes = 0 if f32_scratch is None else f32_scratch.numel() * f32_scratch.element_size()
    return moe_ep_rows(int(rows), _ptr(offsets), _ptr(x), _ptr(h1), _ptr(h3), _ptr(a), _ptr(y),
                       _ptr(dy), _ptr(dh1), _ptr(dh3), _ptr(dx), _ptr(status), _ptr(f32_scratch),
                       nbytes)


def moe_ep_f32_scratch_size(cfg, ep, rows: int) -> int:
    return int(lib().moe_ep_f32_scratch_size(ctypes.byref(cfg), ctypes.byref(ep), int(rows)))


def moe_ep_workspace_size(cfg, ep) -> int:
    return int(lib().moe_ep_workspace_size(ctypes.byref(cfg), ctypes.byref(ep)))


def moe_ep_buffer_offsets(cfg, ep):
    """Byte offsets of (x_e, y_e, dy_e, dx_e) inside the rank's workspace."""
    out = (c_size_t * 4)()
    _check("moe_ep_buffer_offsets",
           lib().moe_ep_buffer_offsets(ctypes.byref(cfg), ctypes.byref(ep), out))
    return [int(v) for v in out]


def moe_ep_get_routing(cfg, ep, workspace, scores=None, idx=None, gate=None, counts=None,
                       offsets=None, src_tok=None, slot_of=None, stream=None):
    _check("moe_ep_get_routing",
           lib().moe_ep_get_routing(ctypes.byref(cfg), ctypes.byref(ep), _ptr(workspace),
                                    workspace.numel(), _ptr(scores), _ptr(idx), _ptr(gate),
                                    _ptr(counts), _ptr(offsets), _ptr(src_tok), _ptr(slot_of),
                                    _stream(stream)))


def moe_ep_route(cfg, ep, weights, x, score_sum, workspace, stream=None):
    _check("moe_ep_route",
           lib().moe_ep_route(ctypes.byref(cfg), ctypes.byref(ep), ctypes.byref(weights), _ptr(x),
                              _ptr(score_sum), _ptr(workspace), workspace.numel(),
                              _stream(stream)))


def moe_ep_expert_forward(cfg, ep, weights, rows, stream=None):
    _check("moe_ep_expert_forward",
           lib().moe_ep_expert_forward(ctypes.byref(cfg), ctypes.byref(ep), ctypes.byref(weights),
                                       ctypes.byref(rows), _stream(stream)))


def moe_ep_combine(cfg, ep, counts_total, score_sum_total, y_target, d_loss, workspace,
                   stream=None):
    _check("moe_ep_combine",
           lib().moe_ep_combine(ctypes.byref(cfg), ctypes.byref(ep), _ptr(counts_total),
                                _ptr(score_sum_total), _ptr(y_target), _ptr(d_loss),
                                _ptr(workspace), workspace.numel(), _stream(stream)))


def moe_ep_expert_backward(cfg, ep, params, rows, lr, stream=None):
    _check("moe_ep_expert_backward",
           lib().moe_ep_expert_backward(ctypes.byref(cfg), ctypes.byref(ep), ctypes.byref(params),
                                        ctypes.byref(rows), float(lr), _stream(stream)))


def moe_ep_router_backward(cfg, ep, w_gate, x, dw_gate_part, dx, workspace, stream=None):
    _check("moe_ep_router_backward",
           lib().moe_ep_router_backward(ctypes.byref(cfg), ctypes.byref(ep), _ptr(w_gate), _ptr(x),
                                        _ptr(dw_gate_part), _ptr(dx), _ptr(workspace),
                                        workspace.numel(), _stream(stream)))


def moe_ep_router_update(cfg, w_gate, dw_gate, lr, stream=None):
    _check("moe_ep_router_update",
           lib().moe_ep_router_update(ctypes.byref(cfg), _ptr(w_gate), _ptr(dw_gate), float(lr),
                                      _stream(stream)))


def moe_build_flags() -> int:
    return int(lib().moe_build_flags())


GEMM_CUDA_CORES, GEMM_TENSOR_BF16, GEMM_TENSOR_F32X3 = 0, 1, 2


def moe_expert_gemm_path(cfg) -> int:
    return int(lib().moe_expert_gemm_path(ctypes.byref(cfg)))


def moe_debug_poke_routing(cfg, workspace, field: int, index: int, value: int, stream=None):
    """Write one routing entry (field 0 idx, 1 slot_of) of the last forward's
    state: the MOE_DEBUG variant's fault injection (the release library
    refuses)."""
    _check("moe_debug_poke_routing",
           lib().moe_debug_poke_routing(ctypes.byref(cfg), _ptr(workspace), workspace.numel(),
                                        int(field), int(index), int(value), _stream(stream)))
