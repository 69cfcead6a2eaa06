"""Float64 CPU oracle for one training step of a sparse top-k MoE layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  The product path (the
CUDA library and its binding) never calls it and shares no code with it.

It is the plain definition of every step, written out in numpy float64 in the
order the course "Trainable MoE in CUDA" layers the method (Parts 1-7):

* Part 1, "CUDA Building Blocks": matmuls, bias add / bias reduction,
  activations (ReLU, GELU with the tanh approximation, SwiGLU) and the
  row-wise softmax, each with its backward.
* Part 2, "Top-K Gating Utilities": the k largest gate values per token and
  their renormalisation to a distribution, with its backward.
* Part 3, "Router": gate matmul -> probabilities -> top-k -> gradient to the
  gate weights.  The sigmoid, group-limited variant follows "AI Infra Kernel
  Lab", section "Project status" (grouped Top-K gate) and the notes under
  "DeepSeek whole-layer MoE forward": exact score ties go to the smaller group
  or expert id; an optional correction bias changes which experts are chosen
  but not the routing weights or their gradients.
* Part 4, "Token Dispatch and Combine": per-expert counts, slot offsets,
  gather into per-expert buffers, scatter of gradients back, gate-weighted
  combine and its backward.
* Part 5, "Expert MLP Forward and Backward" (and the lesson "Define Expert Mlp
  Forward And Backward"): the two-layer expert MLP on each expert's slice of
  tokens and its backward for inputs, weights and biases.  The SwiGLU form is
  W2(SiLU(W1 x) * W3 x) ("AI Infra Kernel Lab", "Numerical contracts").
* Part 6, "Load Balancing Auxiliary Loss": dispatch fractions, mean router
  probabilities, the aux loss and its gradient to router probabilities.
* Part 7, "Loss, Optimizer, and Training Loop": MSE, zero-grad, SGD, and the
  forward / backward / one-step orchestration.
* Shared experts ("AI Infra Kernel Lab", notes on the distributed validator):
  one SwiGLU branch of hidden width n_shared x F that every token passes
  through, added to the routed output without a gate.

The pages lost their typeset formulas, so each step is the textbook
definition; every reading taken where the pages are silent is marked READING
in the docstring that takes it.  Library primitives (numpy ``@``, ``exp``,
``tanh``, a stable ``argsort``) serve as steps; nothing is blocked, fused or
reordered.  For bf16 workloads the caller passes the bf16-rounded values
widened to float64; no intermediate is rounded.

Parity status: every function here is pinned by tests (closed forms,
invariants, brute force on tiny inputs, textbook reductions, central finite
differences, the first-order SGD prediction).  The one choice the pages leave
open without a pin is the group score of the grouped router (sum of the top-2
scores in a group, or the group maximum): both are implemented and that choice
is "parity unpinned".
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

ACTS = ("relu", "gelu_tanh", "swiglu")
SCORES = ("softmax", "sigmoid")


@dataclasses.dataclass(frozen=True)
class OracleConfig:
    T: int
    D: int
    F: int
    E: int
    k: int
    act: str = "relu"
    score: str = "softmax"
    n_groups: int = 1
    topk_groups: int = 1
    group_score: str = "top2_sum"   # or "max"  (parity unpinned choice)
    has_bias: bool = True
    aux_alpha: float = 0.0
    capacity_factor: float = 0.0    # 0: no expert capacity (nothing dropped)


# ---------------------------------------------------------------- Part 1 ---

def softmax_rows(logits: np.ndarray) -> np.ndarray:
    """Row softmax with max subtraction (the course article's advice on
    stability: "Make mathematical equivalence survive finite precision")."""
    m = np.max(logits, axis=1, keepdims=True)
    z = np.exp(logits - m)
    return z / np.sum(z, axis=1, keepdims=True)


def softmax_rows_backward(p: np.ndarray, dp: np.ndarray) -> np.ndarray:
    """dl = p * (dp - <dp, p>) per row."""
    inner = np.sum(dp * p, axis=1, keepdims=True)
    return p * (dp - inner)


def sigmoid(logits: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-logits))


def sigmoid_backward(s: np.ndarray, ds: np.ndarray) -> np.ndarray:
    return ds * s * (1.0 - s)


_GELU_C = np.sqrt(2.0 / np.pi)
_GELU_A = 0.044715


def act_forward(act: str, h: np.ndarray) -> np.ndarray:
    """ReLU, or GELU with the tanh approximation 0.5 h (1 + tanh(c (h + a h^3)))."""
    if act == "relu":
        return np.maximum(h, 0.0)
    if act == "gelu_tanh":
        u = _GELU_C * (h + _GELU_A * h ** 3)
        return 0.5 * h * (1.0 + np.tanh(u))
    raise ValueError(act)


def act_derivative(act: str, h: np.ndarray) -> np.ndarray:
    """d act / d h in closed form (ReLU: 1[h > 0])."""
    if act == "relu":
        return (h > 0.0).astype(np.float64)
    if act == "gelu_tanh":
        u = _GELU_C * (h + _GELU_A * h ** 3)
        t = np.tanh(u)
        du = _GELU_C * (1.0 + 3.0 * _GELU_A * h ** 2)
        return 0.5 * (1.0 + t) + 0.5 * h * (1.0 - t * t) * du
    raise ValueError(act)


def silu(h: np.ndarray) -> np.ndarray:
    return h * sigmoid(h)


def silu_derivative(h: np.ndarray) -> np.ndarray:
    s = sigmoid(h)
    return s * (1.0 + h * (1.0 - s))


# ---------------------------------------------------------------- Part 2 ---

def _order_desc(keys: np.ndarray) -> np.ndarray:
    """Indices of ``keys`` (one row) ordered by descending key, equal keys by
    ascending index: a stable sort on the negated key."""
    return np.argsort(-keys, kind="stable")


def select_topk(scores: np.ndarray, k: int) -> np.ndarray:
    """The k largest scores of every token, in descending score order; equal
    scores go to the smaller expert id.  Comparisons are exact, so the result
    does not depend on the precision the scores are held in."""
    T, E = scores.shape
    if not 1 <= k <= E:
        raise ValueError("k out of range")
    idx = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        idx[t] = _order_desc(scores[t])[:k]
    return idx


def group_scores(scores: np.ndarray, n_groups: int, mode: str = "top2_sum") -> np.ndarray:
    """Score of each of ``n_groups`` groups of contiguous experts.

    READING: the pages name a group-limited (DeepSeek-style) selector but not
    its group score.  Default: sum of the two largest scores in the group (one
    score when a group holds a single expert); ``mode="max"`` takes the group
    maximum.  The sum is taken in the dtype of ``scores`` so that a float32
    score tensor gives the same float32 group scores a float32 kernel does.
    """
    T, E = scores.shape
    if E % n_groups:
        raise ValueError("E must be a multiple of n_groups")
    per = E // n_groups
    g = scores.reshape(T, n_groups, per)
    srt = -np.sort(-g, axis=2)   # descending within each group
    if mode == "max" or per == 1:
        return srt[:, :, 0].copy()
    if mode == "top2_sum":
        return srt[:, :, 0] + srt[:, :, 1]
    raise ValueError(mode)


def select_grouped_topk(scores: np.ndarray, k: int, n_groups: int, topk_groups: int,
                        mode: str = "top2_sum") -> np.ndarray:
    """Group-limited top-k: keep the ``topk_groups`` best groups (equal group
    scores go to the smaller group id), then the k best experts inside the kept
    groups (equal scores go to the smaller expert id), in descending score."""
    T, E = scores.shape
    per = E // n_groups
    if not (1 <= topk_groups <= n_groups) or k > topk_groups * per:
        raise ValueError("group limits out of range")
    gs = group_scores(scores, n_groups, mode)
    idx = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        kept = _order_desc(gs[t])[:topk_groups]
        allowed = np.zeros(E, dtype=bool)
        for gidx in kept:
            allowed[gidx * per:(gidx + 1) * per] = True
        cand = np.flatnonzero(allowed)               # ascending ids
        order = _order_desc(scores[t, cand])
        idx[t] = cand[order[:k]]
    return idx


def renormalize(scores: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """g_tj = s_{t, idx_tj} / sum_j' s_{t, idx_tj'} (no extra scale factor)."""
    sel = np.take_along_axis(scores, idx.astype(np.int64), axis=1)
    return sel / np.sum(sel, axis=1, keepdims=True)


def renormalize_backward(scores: np.ndarray, idx: np.ndarray, gate: np.ndarray,
                         dgate: np.ndarray) -> np.ndarray:
    """Gradient of the renormalised gates with respect to the full score
    tensor: (dg_i - sum_j dg_j g_j) / S on the selected entries, 0 elsewhere."""
    sel = np.take_along_axis(scores, idx.astype(np.int64), axis=1)
    S = np.sum(sel, axis=1, keepdims=True)
    inner = np.sum(dgate * gate, axis=1, keepdims=True)
    dsel = (dgate - inner) / S
    ds = np.zeros_like(scores, dtype=np.float64)
    T = scores.shape[0]
    for t in range(T):
        for j in range(idx.shape[1]):
            ds[t, idx[t, j]] += dsel[t, j]
    return ds


# ---------------------------------------------------------------- Part 3 ---

def router_logits(x: np.ndarray, w_gate: np.ndarray,
                  logit_bias: Optional[np.ndarray] = None) -> np.ndarray:
    """logits = x W_g^T.  READING: the router has no trainable bias; a fixed
    workload logit bias, when given, is added before the score."""
    logits = x @ w_gate.T
    if logit_bias is not None:
        logits = logits + logit_bias[None, :]
    return logits


def router_scores(cfg: OracleConfig, logits: np.ndarray) -> np.ndarray:
    if cfg.score == "softmax":
        return softmax_rows(logits)
    if cfg.score == "sigmoid":
        return sigmoid(logits)
    raise ValueError(cfg.score)


def selection_keys(scores: np.ndarray, corr_bias: Optional[np.ndarray] = None) -> np.ndarray:
    """Keys the selection ranks: the scores, plus a per-expert correction bias
    when one is given ("AI Infra Kernel Lab": the DeepSeek gate's correction
    bias chooses experts only; the routing weights and their gradients come
    from the unbiased scores).  The sum is taken in the dtype of ``scores``, so
    float32 scores give the float32 keys a float32 kernel forms."""
    if corr_bias is None:
        return scores
    return scores + np.asarray(corr_bias).astype(scores.dtype)[None, :]


def route(cfg: OracleConfig, scores: np.ndarray,
          corr_bias: Optional[np.ndarray] = None) -> np.ndarray:
    """Top-k (or group-limited top-k) selection on the score tensor, or on
    score + correction bias (group scores then come from the biased keys)."""
    keys = selection_keys(scores, corr_bias)
    if cfg.n_groups > 1:
        return select_grouped_topk(keys, cfg.k, cfg.n_groups, cfg.topk_groups,
                                   cfg.group_score)
    return select_topk(keys, cfg.k)


# ---------------------------------------------------------------- Part 4 ---

def expert_capacity(cfg: "OracleConfig") -> Optional[int]:
    """Rows an expert may process, or None without a capacity factor.

    READING: the pages name a capacity factor for dropping or padding tokens
    ("AI Infra Kernel Lab", the distributed validator) but give no formula;
    the plainest reading is the usual one, C = ceil(cf * T * k / E)."""
    if cfg.capacity_factor <= 0:
        return None
    return int(math.ceil(cfg.capacity_factor * cfg.T * cfg.k / cfg.E))


def dispatch(idx: np.ndarray, E: int, capacity: Optional[int] = None):
    """Per-expert counts, exclusive-scan offsets and the stable slot map.

    rank(t, j) = #{(t', j') before (t, j) in token order routed to e};
    READING: rows of one expert keep ascending token order (the pages' own
    packing order is atomic and unspecified).  With a capacity C an expert
    keeps the assignments of rank < C (the first C in token order) and drops
    the rest (READING: drop rather than pad, no re-routing).  Returns
    ``counts [E]`` (routed assignments, before any drop), ``offsets [E+1]``
    (exclusive scan of the kept counts), ``src_tok`` / ``src_j`` (slot ->
    token / position in its top-k list, kept slots only) and ``slot_of [T, k]``
    (-1 for a dropped assignment).
    """
    T, k = idx.shape
    counts = np.zeros(E, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            counts[idx[t, j]] += 1
    kept = counts if capacity is None else np.minimum(counts, capacity)
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + kept[e]
    R = int(offsets[E])
    src_tok = np.empty(R, dtype=np.int64)
    src_j = np.empty(R, dtype=np.int64)
    slot_of = np.empty((T, k), dtype=np.int64)
    rank = np.zeros(E, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            r = rank[e]
            rank[e] += 1
            if r < kept[e]:
                s = offsets[e] + r
                src_tok[s] = t
                src_j[s] = j
                slot_of[t, j] = s
            else:
                slot_of[t, j] = -1
    return counts, offsets, src_tok, src_j, slot_of


def gather_rows(x: np.ndarray, src_tok: np.ndarray) -> np.ndarray:
    """Expert-major copy: Xe[s] = x[src_tok[s]]."""
    return x[src_tok]


def combine(ye: np.ndarray, gate: np.ndarray, slot_of: np.ndarray) -> np.ndarray:
    """Y[t] = sum_j g_tj Ye[slot(t, j)], summed in j order; a dropped
    assignment (slot -1) contributes nothing (READING: the gates are not
    renormalised over the kept experts)."""
    T, k = gate.shape
    y = np.zeros((T, ye.shape[1]), dtype=np.float64)
    for j in range(k):
        kept = slot_of[:, j] >= 0
        y[kept] += gate[kept, j:j + 1] * ye[slot_of[kept, j]]
    return y


def combine_backward(dy: np.ndarray, ye: np.ndarray, gate: np.ndarray,
                     slot_of: np.ndarray):
    """dYe[slot(t,j)] = g_tj dY[t];  dg_tj = <dY[t], Ye[slot(t,j)]> (0 for a
    dropped assignment)."""
    T, k = gate.shape
    dye = np.zeros_like(ye, dtype=np.float64)
    dgate = np.zeros((T, k), dtype=np.float64)
    for j in range(k):
        kept = slot_of[:, j] >= 0
        rows = slot_of[kept, j]
        dye[rows] = gate[kept, j:j + 1] * dy[kept]
        dgate[kept, j] = np.sum(dy[kept] * ye[rows], axis=1)
    return dye, dgate


def scatter_back(dxe: np.ndarray, slot_of: np.ndarray) -> np.ndarray:
    """dX[t] = sum_j dXe[slot(t, j)] (j order, kept assignments only)."""
    T, k = slot_of.shape
    dx = np.zeros((T, dxe.shape[1]), dtype=np.float64)
    for j in range(k):
        kept = slot_of[:, j] >= 0
        dx[kept] += dxe[slot_of[kept, j]]
    return dx


# ---------------------------------------------------------------- Part 5 ---

def expert_forward(cfg: OracleConfig, e: int, xe: np.ndarray, w: dict) -> dict:
    """Two-layer MLP of expert e on its rows ``xe [n, D]``.

    ReLU / GELU:  H = xe W1_e^T + b1_e;  A = act(H);  Ye = A W2_e^T + b2_e.
    SwiGLU:       H1 = xe W1_e^T, H3 = xe W3_e^T;  A = SiLU(H1) * H3;
                  Ye = A W2_e^T (no biases).
    """
    out = {}
    if cfg.act == "swiglu":
        if cfg.has_bias:
            raise ValueError("the SwiGLU experts carry no biases")
        h1 = xe @ w["w1"][e].T
        h3 = xe @ w["w3"][e].T
        a = silu(h1) * h3
        out.update(h1=h1, h3=h3)
    else:
        h = xe @ w["w1"][e].T
        if cfg.has_bias:
            h = h + w["b1"][e]
        a = act_forward(cfg.act, h)
        out.update(h=h)
    ye = a @ w["w2"][e].T
    if cfg.has_bias:
        ye = ye + w["b2"][e]
    out.update(a=a, ye=ye)
    return out


def expert_backward(cfg: OracleConfig, e: int, xe: np.ndarray, fwd: dict,
                    dye: np.ndarray, w: dict) -> dict:
    """Backward of expert e: dXe, dW1, dW3 (SwiGLU), dW2, db1, db2.  An expert
    with no rows gets exact zeros."""
    a = fwd["a"]
    dw2 = dye.T @ a
    db2 = np.sum(dye, axis=0)
    da = dye @ w["w2"][e]
    if cfg.act == "swiglu":
        h1, h3 = fwd["h1"], fwd["h3"]
        dh1 = da * h3 * silu_derivative(h1)
        dh3 = da * silu(h1)
        dxe = dh1 @ w["w1"][e] + dh3 @ w["w3"][e]
        out = dict(dxe=dxe, dw1=dh1.T @ xe, dw3=dh3.T @ xe, dw2=dw2,
                   db1=np.sum(dh1, axis=0), db2=db2)
    else:
        dh = da * act_derivative(cfg.act, fwd["h"])
        dxe = dh @ w["w1"][e]
        out = dict(dxe=dxe, dw1=dh.T @ xe, dw2=dw2, db1=np.sum(dh, axis=0), db2=db2)
    return out


def shared_forward(x: np.ndarray, w: dict) -> dict:
    """Shared experts: one SwiGLU MLP that every token passes through, added to
    the routed output without a gate ("AI Infra Kernel Lab": the replicated
    shared branch is one SwiGLU whose hidden width is n_shared times the
    expert hidden width).  H1 = x Ws1^T, H3 = x Ws3^T, A = SiLU(H1) * H3,
    Ys = A Ws2^T."""
    h1 = x @ w["ws1"].T
    h3 = x @ w["ws3"].T
    a = silu(h1) * h3
    return dict(h1=h1, h3=h3, a=a, ys=a @ w["ws2"].T)


def shared_backward(x: np.ndarray, fwd: dict, dy: np.ndarray, w: dict) -> dict:
    """The shared branch receives the whole dY: dWs2 = dY^T A, dA = dY Ws2,
    the SwiGLU backward, dWs1 = dH1^T x, dWs3 = dH3^T x, and its dX term."""
    da = dy @ w["ws2"]
    dh1 = da * fwd["h3"] * silu_derivative(fwd["h1"])
    dh3 = da * silu(fwd["h1"])
    return dict(dws1=dh1.T @ x, dws3=dh3.T @ x, dws2=dy.T @ fwd["a"],
                dx=dh1 @ w["ws1"] + dh3 @ w["ws3"])


# ---------------------------------------------------------------- Part 6 ---

def aux_loss(counts: np.ndarray, scores: np.ndarray, k: int):
    """f_e = c_e / (T k), P_e = mean_t s_te, aux = E sum_e f_e P_e.

    READING: f is normalised by the T k routed rows so that aux is exactly 1
    under uniform routing; P averages the full (pre-top-k) score tensor.
    Returns (aux, f, P).
    """
    T, E = scores.shape
    f = counts.astype(np.float64) / float(T * k)
    P = np.mean(scores, axis=0)
    return float(E * np.sum(f * P)), f, P


def aux_loss_score_grad(f: np.ndarray, T: int) -> np.ndarray:
    """d aux / d s_te = E f_e / T for every token (counts carry no gradient)."""
    E = f.shape[0]
    return E * f / float(T)


# ---------------------------------------------------------------- Part 7 ---

def mse_loss(y: np.ndarray, target: np.ndarray):
    """READING: mean over all T*D elements, no 1/2 factor.  Returns (L, dY)."""
    diff = y - target
    n = float(diff.size)
    return float(np.sum(diff * diff) / n), 2.0 * diff / n


def forward(cfg: OracleConfig, w: dict, x: np.ndarray,
            idx: Optional[np.ndarray] = None) -> dict:
    """Router, dispatch, experts and combine.  ``idx`` forces a routing (used
    only after that routing has been validated against this oracle's own)."""
    logits = router_logits(x, w["w_gate"], w.get("logit_bias"))
    scores = router_scores(cfg, logits)
    if idx is None:
        idx = route(cfg, scores, w.get("corr_bias"))
    gate = renormalize(scores, idx)      # unbiased scores, with or without a correction bias
    counts, offsets, src_tok, src_j, slot_of = dispatch(idx, cfg.E, expert_capacity(cfg))
    xe = gather_rows(x, src_tok)
    R = xe.shape[0]
    ye = np.zeros((R, cfg.D), dtype=np.float64)
    experts = []
    for e in range(cfg.E):
        lo, hi = offsets[e], offsets[e + 1]
        fe = expert_forward(cfg, e, xe[lo:hi], w)
        ye[lo:hi] = fe["ye"]
        experts.append(fe)
    y = combine(ye, gate, slot_of)
    shared = None
    if w.get("ws1") is not None:
        shared = shared_forward(x, w)
        y = y + shared["ys"]
    return dict(logits=logits, scores=scores, idx=idx, gate=gate, counts=counts,
                offsets=offsets, src_tok=src_tok, src_j=src_j, slot_of=slot_of,
                xe=xe, ye=ye, experts=experts, y=y, shared=shared)


def backward(cfg: OracleConfig, w: dict, x: np.ndarray, st: dict,
             dy: np.ndarray) -> dict:
    """Gradients of L = L_task + alpha * aux, given dY = dL_task/dY."""
    dye, dgate = combine_backward(dy, st["ye"], st["gate"], st["slot_of"])
    offsets = st["offsets"]
    R = st["xe"].shape[0]
    dxe = np.zeros((R, cfg.D), dtype=np.float64)
    g = dict(dw1=np.zeros_like(w["w1"], dtype=np.float64),
             dw2=np.zeros_like(w["w2"], dtype=np.float64),
             db1=np.zeros((cfg.E, cfg.F)), db2=np.zeros((cfg.E, cfg.D)))
    if cfg.act == "swiglu":
        g["dw3"] = np.zeros_like(w["w3"], dtype=np.float64)
    for e in range(cfg.E):
        lo, hi = offsets[e], offsets[e + 1]
        be = expert_backward(cfg, e, st["xe"][lo:hi], st["experts"][e], dye[lo:hi], w)
        dxe[lo:hi] = be["dxe"]
        for key in ("dw1", "dw2", "db1", "db2") + (("dw3",) if cfg.act == "swiglu" else ()):
            g[key][e] = be[key]
    dx = scatter_back(dxe, st["slot_of"])
    if st.get("shared") is not None:
        sb = shared_backward(x, st["shared"], dy, w)
        dx = dx + sb["dx"]
        g.update(dws1=sb["dws1"], dws3=sb["dws3"], dws2=sb["dws2"])
    # router: renormalisation backward, aux gradient, score backward
    ds = renormalize_backward(st["scores"], st["idx"], st["gate"], dgate)
    if cfg.aux_alpha != 0.0:
        _, f, _ = aux_loss(st["counts"], st["scores"], cfg.k)
        ds = ds + cfg.aux_alpha * aux_loss_score_grad(f, cfg.T)[None, :]
    if cfg.score == "softmax":
        dl = softmax_rows_backward(st["scores"], ds)
    else:
        dl = sigmoid_backward(st["scores"], ds)
    g["dw_gate"] = dl.T @ x
    dx = dx + dl @ w["w_gate"]
    g["dx"] = dx
    g.update(dye=dye, dgate=dgate, dxe=dxe, dlogits=dl)
    if not cfg.has_bias:
        g["db1"] = None
        g["db2"] = None
    return g


def losses(cfg: OracleConfig, st: dict, target: np.ndarray):
    """(L_mse, aux, dY)."""
    l_mse, dy = mse_loss(st["y"], target)
    aux, _, _ = aux_loss(st["counts"], st["scores"], cfg.k)
    return l_mse, aux, dy


def total_loss(cfg: OracleConfig, w: dict, x: np.ndarray, target: np.ndarray,
               idx: Optional[np.ndarray] = None) -> float:
    st = forward(cfg, w, x, idx)
    l_mse, aux, _ = losses(cfg, st, target)
    return l_mse + cfg.aux_alpha * aux


PARAM_KEYS = ("w_gate", "w1", "w3", "w2", "b1", "b2", "ws1", "ws3", "ws2")


def sgd(w: dict, grads: dict, lr: float) -> dict:
    """theta <- theta - lr * grad for the router and expert parameters."""
    out = dict(w)
    for key in PARAM_KEYS:
        if w.get(key) is not None and grads.get("d" + key) is not None:
            out[key] = w[key] - lr * grads["d" + key]
    return out


def train_step(cfg: OracleConfig, w: dict, x: np.ndarray, target: np.ndarray,
               lr: float, idx: Optional[np.ndarray] = None):
    """One step: forward, losses, backward, SGD.  Returns (new weights,
    (L_mse, aux), forward state, gradients)."""
    st = forward(cfg, w, x, idx)
    l_mse, aux, dy = losses(cfg, st, target)
    grads = backward(cfg, w, x, st, dy)
    return sgd(w, grads, lr), (l_mse, aux), st, grads
