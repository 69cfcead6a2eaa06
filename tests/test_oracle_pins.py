"""Pins of the float64 oracle against things other than itself.

Each test checks the oracle against a closed form, an invariant, brute force
on tiny inputs, a textbook/library routine, central finite differences or the
first-order SGD prediction, chosen so that a dropped term, a wrong sign or
index, or a transposed operand fails at least one of them.  CPU only.
"""

import itertools
import math

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O

pytestmark = []


# ------------------------------------------------------------------ scores ---

def test_softmax_closed_form():
    # logits 0, ln2, ln3 -> probabilities 1/6, 2/6, 3/6 exactly
    l = np.array([[0.0, math.log(2.0), math.log(3.0)]])
    p = O.softmax_rows(l)
    np.testing.assert_allclose(p, [[1 / 6, 2 / 6, 3 / 6]], rtol=1e-15, atol=0)


def test_softmax_invariants_and_library():
    rng = np.random.default_rng(1)
    l = rng.normal(size=(7, 11)) * 5
    p = O.softmax_rows(l)
    np.testing.assert_allclose(p.sum(1), 1.0, rtol=0, atol=1e-15)
    np.testing.assert_allclose(O.softmax_rows(l + 123.25), p, rtol=1e-13, atol=1e-16)
    ref = torch.softmax(torch.from_numpy(l), dim=1).numpy()
    np.testing.assert_allclose(p, ref, rtol=1e-14, atol=1e-17)
    # a huge logit must not overflow (max subtraction)
    p2 = O.softmax_rows(np.array([[1000.0, 0.0]]))
    assert np.isfinite(p2).all() and p2[0, 0] == pytest.approx(1.0)


def test_softmax_backward_vs_autograd():
    rng = np.random.default_rng(2)
    l = rng.normal(size=(5, 6))
    dp = rng.normal(size=(5, 6))
    lt = torch.from_numpy(l).requires_grad_(True)
    (torch.softmax(lt, 1) * torch.from_numpy(dp)).sum().backward()
    np.testing.assert_allclose(O.softmax_rows_backward(O.softmax_rows(l), dp),
                               lt.grad.numpy(), rtol=1e-12, atol=1e-15)


def test_sigmoid_closed_form_and_backward():
    s = O.sigmoid(np.array([0.0, math.log(3.0), -math.log(3.0)]))
    np.testing.assert_allclose(s, [0.5, 0.75, 0.25], rtol=1e-15)
    ds = O.sigmoid_backward(s, np.ones(3))
    np.testing.assert_allclose(ds, [0.25, 0.1875, 0.1875], rtol=1e-14)


def test_activations_match_library():
    h = np.linspace(-6, 6, 1001)
    ht = torch.from_numpy(h)
    np.testing.assert_allclose(O.act_forward("relu", h), torch.relu(ht).numpy(), atol=0)
    np.testing.assert_allclose(O.act_forward("gelu_tanh", h),
                               torch.nn.functional.gelu(ht, approximate="tanh").numpy(),
                               rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(O.silu(h), torch.nn.functional.silu(ht).numpy(),
                               rtol=1e-14, atol=1e-16)
    # derivatives against autograd
    for name, fn in (("gelu_tanh", lambda v: torch.nn.functional.gelu(v, approximate="tanh")),):
        v = ht.clone().requires_grad_(True)
        fn(v).sum().backward()
        np.testing.assert_allclose(O.act_derivative(name, h), v.grad.numpy(),
                                   rtol=1e-12, atol=1e-14)
    v = ht.clone().requires_grad_(True)
    torch.nn.functional.silu(v).sum().backward()
    np.testing.assert_allclose(O.silu_derivative(h), v.grad.numpy(), rtol=1e-12, atol=1e-15)
    hr = np.array([-1.0, -1e-9, 1e-9, 2.0])
    np.testing.assert_array_equal(O.act_derivative("relu", hr), [0, 0, 1, 1])


# ------------------------------------------------------------------- top-k ---

def _dominates(si, i, sj, j):
    """(s_i, i) beats (s_j, j): larger score, equal score -> smaller id."""
    return si > sj or (si == sj and i < j)


def _brute_topk_set(s, k):
    E = len(s)
    winners = []
    for S in itertools.combinations(range(E), k):
        rest = [j for j in range(E) if j not in S]
        if all(_dominates(s[i], i, s[j], j) for i in S for j in rest):
            winners.append(set(S))
    assert len(winners) == 1
    return winners[0]


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(3)
    for E in range(1, 7):
        for k in range(1, E + 1):
            s = rng.integers(0, 3, size=(40, E)).astype(np.float64)  # many ties
            idx = O.select_topk(s, k)
            for t in range(40):
                assert set(idx[t].tolist()) == _brute_topk_set(s[t], k)
                # order: descending score, ties by ascending id
                for a, b in zip(idx[t][:-1], idx[t][1:]):
                    assert _dominates(s[t, a], a, s[t, b], b)


def test_topk_all_equal_selects_smallest_ids():
    idx = O.select_topk(np.full((3, 8), 0.125), 3)
    np.testing.assert_array_equal(idx, [[0, 1, 2]] * 3)


def test_topk_permutation_metamorphic():
    rng = np.random.default_rng(4)
    s = rng.normal(size=(50, 9))            # distinct scores
    perm = rng.permutation(9)
    idx = O.select_topk(s, 4)
    idx_p = O.select_topk(s[:, perm], 4)   # column c of the permuted = expert perm[c]
    np.testing.assert_array_equal(perm[idx_p], idx)


def _brute_grouped(s, k, G, kg, mode):
    E = len(s)
    per = E // G
    grp = []
    for g in range(G):
        v = sorted(s[g * per:(g + 1) * per], reverse=True)
        grp.append(v[0] + v[1] if (mode == "top2_sum" and per > 1) else v[0])
    win_g = [set(S) for S in itertools.combinations(range(G), kg)
             if all(_dominates(grp[a], a, grp[b], b) for a in S for b in range(G) if b not in S)]
    assert len(win_g) == 1
    allowed = [e for e in range(E) if e // per in win_g[0]]
    win = [set(S) for S in itertools.combinations(allowed, k)
           if all(_dominates(s[a], a, s[b], b) for a in S for b in allowed if b not in S)]
    assert len(win) == 1
    return win[0]


@pytest.mark.parametrize("mode", ["top2_sum", "max"])
def test_grouped_topk_brute_force(mode):
    rng = np.random.default_rng(5)
    E, G, kg, k = 8, 4, 2, 3
    s = rng.integers(0, 4, size=(60, E)).astype(np.float64) / 4.0
    idx = O.select_grouped_topk(s, k, G, kg, mode)
    for t in range(60):
        assert set(idx[t].tolist()) == _brute_grouped(s[t], k, G, kg, mode)
        for a, b in zip(idx[t][:-1], idx[t][1:]):
            assert _dominates(s[t, a], a, s[t, b], b)


def test_grouped_topk_group_score_distinguishes_modes():
    # group 0: (0.9, 0.1) -> sum 1.0, max 0.9;  group 1: (0.6, 0.6) -> sum 1.2, max 0.6
    s = np.array([[0.9, 0.1, 0.6, 0.6]])
    assert O.select_grouped_topk(s, 1, 2, 1, "top2_sum").tolist() == [[2]]
    assert O.select_grouped_topk(s, 1, 2, 1, "max").tolist() == [[0]]


def test_grouped_topk_reduces_to_plain():
    rng = np.random.default_rng(6)
    s = rng.random((30, 16))
    plain = O.select_topk(s, 5)
    np.testing.assert_array_equal(O.select_grouped_topk(s, 5, 1, 1), plain)
    np.testing.assert_array_equal(O.select_grouped_topk(s, 5, 4, 4), plain)


def test_grouped_group_sum_in_float32():
    # two float32 scores whose float32 sum differs from the float64 sum
    a = np.float32(0.1)
    b = np.float32(0.2)
    s = np.array([[a, b]], dtype=np.float32)
    gs = O.group_scores(s, 1)
    assert gs.dtype == np.float32 and gs[0, 0] == np.float32(a + b)


# ------------------------------------------------------------------ renorm ---

def test_renormalize_closed_forms():
    rng = np.random.default_rng(7)
    p = O.softmax_rows(rng.normal(size=(20, 6)))
    idx = O.select_topk(p, 3)
    g = O.renormalize(p, idx)
    np.testing.assert_allclose(g.sum(1), 1.0, atol=1e-15)
    np.testing.assert_array_equal(O.renormalize(p, O.select_topk(p, 1)), 1.0)
    full = O.select_topk(p, 6)
    np.testing.assert_allclose(O.renormalize(p, full), np.take_along_axis(p, full, 1),
                               rtol=1e-14)
    # hand case: selected 0.3 and 0.1 -> 0.75, 0.25
    g2 = O.renormalize(np.array([[0.3, 0.1, 0.05]]), np.array([[0, 1]]))
    np.testing.assert_allclose(g2, [[0.75, 0.25]], rtol=1e-15)


def test_renormalize_backward_vs_autograd():
    rng = np.random.default_rng(8)
    s = rng.random((6, 5)) + 0.1
    idx = O.select_topk(s, 3)
    dg = rng.normal(size=(6, 3))
    st = torch.from_numpy(s).requires_grad_(True)
    sel = torch.gather(st, 1, torch.from_numpy(idx.astype(np.int64)))
    (sel / sel.sum(1, keepdim=True) * torch.from_numpy(dg)).sum().backward()
    g = O.renormalize(s, idx)
    np.testing.assert_allclose(O.renormalize_backward(s, idx, g, dg), st.grad.numpy(),
                               rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------- dispatch ---

def test_dispatch_invariants():
    rng = np.random.default_rng(9)
    T, E, k = 37, 6, 3
    p = O.softmax_rows(rng.normal(size=(T, E)))
    idx = O.select_topk(p, k)
    counts, off, src_tok, src_j, slot_of = O.dispatch(idx, E)
    assert counts.sum() == T * k
    assert off[0] == 0 and off[-1] == T * k
    np.testing.assert_array_equal(np.diff(off), counts)
    # counts by an independent method
    np.testing.assert_array_equal(counts, np.bincount(idx.ravel(), minlength=E))
    # bijection onto (t, j)
    pairs = set(zip(src_tok.tolist(), src_j.tolist()))
    assert len(pairs) == T * k
    for s in range(T * k):
        assert slot_of[src_tok[s], src_j[s]] == s
    for e in range(E):
        seg = src_tok[off[e]:off[e + 1]]
        assert np.all(np.diff(seg) > 0)                     # ascending tokens
        assert np.all(idx[seg, src_j[off[e]:off[e + 1]]] == e)


def test_dispatch_empty_experts():
    idx = np.array([[2, 0], [0, 2], [2, 0]])
    counts, off, src_tok, src_j, slot_of = O.dispatch(idx, 5)
    np.testing.assert_array_equal(counts, [3, 0, 3, 0, 0])
    np.testing.assert_array_equal(off, [0, 3, 3, 6, 6, 6])
    np.testing.assert_array_equal(src_tok, [0, 1, 2, 0, 1, 2])
    np.testing.assert_array_equal(src_j, [1, 0, 1, 0, 1, 0])
    np.testing.assert_array_equal(slot_of, [[3, 0], [1, 4], [5, 2]])


# -------------------------------------------------------- tiny models/grads ---

def _weights(cfg, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    w = dict(w_gate=rng.normal(size=(cfg.E, cfg.D)) * scale,
             w1=rng.normal(size=(cfg.E, cfg.F, cfg.D)) / math.sqrt(cfg.D),
             w2=rng.normal(size=(cfg.E, cfg.D, cfg.F)) / math.sqrt(cfg.F))
    if cfg.act == "swiglu":
        w["w3"] = rng.normal(size=(cfg.E, cfg.F, cfg.D)) / math.sqrt(cfg.D)
    if cfg.has_bias:
        w["b1"] = rng.normal(size=(cfg.E, cfg.F)) * 0.1
        w["b2"] = rng.normal(size=(cfg.E, cfg.D)) * 0.1
    x = rng.normal(size=(cfg.T, cfg.D))
    target = rng.normal(size=(cfg.T, cfg.D))
    return w, x, target


def _torch_dense_mlp(cfg, w, xt, e):
    W1 = torch.from_numpy(w["w1"][e])
    W2 = torch.from_numpy(w["w2"][e])
    b1 = torch.from_numpy(w["b1"][e]) if cfg.has_bias else None
    b2 = torch.from_numpy(w["b2"][e]) if cfg.has_bias else None
    F_ = torch.nn.functional
    if cfg.act == "swiglu":
        h = F_.silu(F_.linear(xt, W1)) * F_.linear(xt, torch.from_numpy(w["w3"][e]))
    elif cfg.act == "relu":
        h = F_.relu(F_.linear(xt, W1, b1))
    else:
        h = F_.gelu(F_.linear(xt, W1, b1), approximate="tanh")
    return F_.linear(h, W2, b2)


@pytest.mark.parametrize("act", ["relu", "gelu_tanh", "swiglu"])
def test_single_expert_is_plain_mlp(act):
    cfg = O.OracleConfig(T=9, D=5, F=7, E=1, k=1, act=act, has_bias=(act != "swiglu"))
    w, x, _ = _weights(cfg, 10)
    st = O.forward(cfg, w, x)
    ref = _torch_dense_mlp(cfg, w, torch.from_numpy(x), 0).numpy()
    np.testing.assert_allclose(st["y"], ref, rtol=1e-12, atol=1e-14)


def test_k_equals_E_is_dense_softmax_mixture():
    cfg = O.OracleConfig(T=11, D=4, F=6, E=3, k=3, act="gelu_tanh", has_bias=True)
    w, x, _ = _weights(cfg, 11)
    st = O.forward(cfg, w, x)
    xt = torch.from_numpy(x)
    p = torch.softmax(xt @ torch.from_numpy(w["w_gate"]).T, 1)
    ref = sum(p[:, e:e + 1] * _torch_dense_mlp(cfg, w, xt, e) for e in range(3))
    np.testing.assert_allclose(st["y"], ref.numpy(), rtol=1e-12, atol=1e-14)


def test_aux_closed_forms():
    T, E, k = 12, 4, 2
    # W_g = 0 -> p = 1/E -> aux = sum_e f_e = 1 whatever the routing
    cfg = O.OracleConfig(T=T, D=3, F=4, E=E, k=k, aux_alpha=0.01)
    w, x, tgt = _weights(cfg, 12)
    w["w_gate"] = np.zeros_like(w["w_gate"])
    st = O.forward(cfg, w, x)
    aux, f, P = O.aux_loss(st["counts"], st["scores"], k)
    assert aux == pytest.approx(1.0, abs=1e-15)
    # perfectly balanced routing with p = 1/E: aux = 1
    idx = np.array([[(2 * t) % E, (2 * t + 1) % E] for t in range(T)])
    counts = np.bincount(idx.ravel(), minlength=E)
    assert O.aux_loss(counts, np.full((T, E), 1.0 / E), k)[0] == pytest.approx(1.0, abs=1e-15)
    # everything on experts {1, 3}, p split 1/2 on them -> aux = E / k
    p = np.zeros((T, E)); p[:, 1] = 0.5; p[:, 3] = 0.5
    counts = np.array([0, T, 0, T])
    assert O.aux_loss(counts, p, k)[0] == pytest.approx(E / k, abs=1e-15)
    # explicit formula on a hand case: E=2, f=(3/4,1/4), P=(0.6,0.4) -> 2*(0.45+0.1)=1.1
    p = np.array([[0.6, 0.4], [0.6, 0.4]])
    assert O.aux_loss(np.array([3, 1]), p, 2)[0] == pytest.approx(1.1, abs=1e-15)


def test_mse_closed_form():
    y = np.array([[1.0, 2.0], [3.0, 4.0]])
    t = np.array([[1.0, 0.0], [0.0, 4.0]])
    L, dy = O.mse_loss(y, t)
    assert L == pytest.approx((4.0 + 9.0) / 4.0)
    np.testing.assert_allclose(dy, [[0.0, 1.0], [1.5, 0.0]])


GRAD_CASES = [
    dict(act="relu", score="softmax", has_bias=True, aux_alpha=0.01),
    dict(act="gelu_tanh", score="softmax", has_bias=True, aux_alpha=0.05),
    dict(act="swiglu", score="softmax", has_bias=False, aux_alpha=0.01),
    dict(act="swiglu", score="sigmoid", has_bias=False, aux_alpha=0.0, E=8,
         n_groups=4, topk_groups=2),
    dict(act="swiglu", score="sigmoid", has_bias=False, aux_alpha=0.02, E=8,
         n_groups=4, topk_groups=2, group_score="max"),
]


def _margin_ok(cfg, w, x):
    st = O.forward(cfg, w, x)
    s = st["scores"]
    for t in range(cfg.T):
        sel = set(st["idx"][t].tolist())
        lo = min(s[t, list(sel)])
        others = [s[t, e] for e in range(cfg.E) if e not in sel]
        if others and lo - max(others) < 1e-3:
            if cfg.n_groups == 1:
                return False
        v = np.sort(s[t])[::-1]
        if np.min(np.abs(np.diff(v))) < 1e-3:
            return False
        if cfg.n_groups > 1:
            gs = np.sort(O.group_scores(s[t:t + 1], cfg.n_groups, cfg.group_score)[0])
            if np.min(np.abs(np.diff(gs))) < 1e-3:
                return False
    for fe in st["experts"]:
        for key in ("h", "h1"):
            if key in fe and fe[key].size and np.min(np.abs(fe[key])) < 1e-3:
                return False
    return True


def _cfg_and_inputs(case, seed0):
    c = dict(T=8, D=4, F=6, E=4, k=2)
    c.update(case)
    cfg = O.OracleConfig(**c)
    for seed in range(seed0, seed0 + 400):
        w, x, tgt = _weights(cfg, seed, scale=1.5)
        if _margin_ok(cfg, w, x):
            return cfg, w, x, tgt
    raise RuntimeError("no input with a routing margin found")


@pytest.mark.parametrize("case", GRAD_CASES)
def test_gradients_central_differences(case):
    cfg, w, x, tgt = _cfg_and_inputs(case, 100)
    st = O.forward(cfg, w, x)
    _, _, dy = O.losses(cfg, st, tgt)
    g = O.backward(cfg, w, x, st, dy)
    h = 1e-6

    def L(wd, xx):
        return O.total_loss(cfg, wd, xx, tgt)

    checks = [(k_, "d" + k_) for k_ in O.PARAM_KEYS if w.get(k_) is not None]
    for key, gkey in checks:
        fd = np.zeros_like(w[key])
        it = np.nditer(w[key], flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            wp = {kk: (vv.copy() if isinstance(vv, np.ndarray) else vv) for kk, vv in w.items()}
            wm = {kk: (vv.copy() if isinstance(vv, np.ndarray) else vv) for kk, vv in w.items()}
            wp[key][i] += h
            wm[key][i] -= h
            fd[i] = (L(wp, x) - L(wm, x)) / (2 * h)
        err = np.max(np.abs(fd - g[gkey])) / max(np.max(np.abs(fd)), 1e-30)
        assert err <= 1e-6, (key, err)
    fd = np.zeros_like(x)
    for i in np.ndindex(x.shape):
        xp = x.copy(); xp[i] += h
        xm = x.copy(); xm[i] -= h
        fd[i] = (L(w, xp) - L(w, xm)) / (2 * h)
    err = np.max(np.abs(fd - g["dx"])) / np.max(np.abs(fd))
    assert err <= 1e-6, ("x", err)


@pytest.mark.parametrize("case", GRAD_CASES[:3])
def test_gradients_vs_dense_autograd(case):
    """The same gradients from torch autograd on an independent dense
    formulation with the routing mask held fixed."""
    cfg, w, x, tgt = _cfg_and_inputs(case, 300)
    st = O.forward(cfg, w, x)
    _, _, dy = O.losses(cfg, st, tgt)
    g = O.backward(cfg, w, x, st, dy)
    tw = {k_: torch.from_numpy(v.copy()).requires_grad_(True)
          for k_, v in w.items() if isinstance(v, np.ndarray)}
    xt = torch.from_numpy(x.copy()).requires_grad_(True)
    mask = torch.zeros(cfg.T, cfg.E, dtype=torch.float64)
    for t in range(cfg.T):
        mask[t, st["idx"][t]] = 1.0
    p = torch.softmax(xt @ tw["w_gate"].T, 1)
    gate = mask * p / (mask * p).sum(1, keepdim=True)
    F_ = torch.nn.functional
    y = 0
    for e in range(cfg.E):
        if cfg.act == "swiglu":
            hh = F_.silu(xt @ tw["w1"][e].T) * (xt @ tw["w3"][e].T)
        else:
            pre = xt @ tw["w1"][e].T + tw["b1"][e]
            hh = F_.relu(pre) if cfg.act == "relu" else F_.gelu(pre, approximate="tanh")
        ye = hh @ tw["w2"][e].T + (tw["b2"][e] if cfg.has_bias else 0)
        y = y + gate[:, e:e + 1] * ye
    mse = ((y - torch.from_numpy(tgt)) ** 2).mean()
    counts = torch.from_numpy(st["counts"].astype(np.float64))
    aux = cfg.E * (counts / (cfg.T * cfg.k) * p.mean(0)).sum()
    (mse + cfg.aux_alpha * aux).backward()
    for key in tw:
        np.testing.assert_allclose(g["d" + key], tw[key].grad.numpy(), rtol=1e-10,
                                   atol=1e-13, err_msg=key)
    np.testing.assert_allclose(g["dx"], xt.grad.numpy(), rtol=1e-10, atol=1e-13)


def test_sgd_first_order_prediction():
    cfg, w, x, tgt = _cfg_and_inputs(GRAD_CASES[1], 500)
    lr = 1e-4
    L0 = O.total_loss(cfg, w, x, tgt)
    w1, (lm, la), st, grads = O.train_step(cfg, w, x, tgt, lr)
    assert lm + cfg.aux_alpha * la == pytest.approx(L0, rel=1e-14)
    L1 = O.total_loss(cfg, w1, x, tgt, st["idx"])
    gn2 = sum(float(np.sum(grads["d" + k_] ** 2)) for k_ in O.PARAM_KEYS
              if w.get(k_) is not None)
    ratio = (L0 - L1) / (lr * gn2)
    assert abs(ratio - 1.0) < 1e-2, ratio


def test_empty_expert_gets_exact_zero_grads():
    cfg = O.OracleConfig(T=6, D=3, F=4, E=4, k=1, act="relu", has_bias=True, aux_alpha=0.01)
    w, x, tgt = _weights(cfg, 13)
    w["w_gate"] = np.zeros_like(w["w_gate"])
    w["w_gate"][0, 0] = 5.0                  # every token picks expert 0 or a tie winner
    st = O.forward(cfg, w, x, idx=np.zeros((6, 1), dtype=np.int32))
    _, _, dy = O.losses(cfg, st, tgt)
    g = O.backward(cfg, w, x, st, dy)
    for e in (1, 2, 3):
        assert np.all(g["dw1"][e] == 0) and np.all(g["dw2"][e] == 0)
        assert np.all(g["db1"][e] == 0) and np.all(g["db2"][e] == 0)


# -------------------------------------------------- correction-bias routing ---
# "AI Infra Kernel Lab": the DeepSeek gate's correction bias chooses the experts
# only; the routing weights (and their gradients) come from the unbiased scores.

def test_corr_bias_zero_and_uniform_shift_change_nothing():
    rng = np.random.default_rng(41)
    s = rng.random((50, 12))
    cfg = O.OracleConfig(T=50, D=1, F=1, E=12, k=3)
    plain = O.route(cfg, s)
    np.testing.assert_array_equal(O.route(cfg, s, np.zeros(12)), plain)
    np.testing.assert_array_equal(O.route(cfg, s, np.full(12, 0.5)), plain)
    cfg_g = O.OracleConfig(T=50, D=1, F=1, E=12, k=3, n_groups=4, topk_groups=2)
    np.testing.assert_array_equal(O.route(cfg_g, s, np.full(12, 0.5)), O.route(cfg_g, s))


def test_corr_bias_brute_force_keys_select_scores_weigh():
    rng = np.random.default_rng(42)
    E, k = 6, 2
    cfg = O.OracleConfig(T=40, D=1, F=1, E=E, k=k)
    s = rng.integers(1, 5, size=(40, E)).astype(np.float64) / 8.0     # ties in s
    b = np.array([0.0, 0.25, -0.125, 0.125, 0.0, 0.375])              # ties in s + b
    idx = O.route(cfg, s, b)
    gate = O.renormalize(s, idx)
    for t in range(40):
        key = s[t] + b
        assert set(idx[t].tolist()) == _brute_topk_set(key, k)
        for a, c in zip(idx[t][:-1], idx[t][1:]):
            assert _dominates(key[a], a, key[c], c)
        sel = idx[t]
        np.testing.assert_allclose(gate[t], s[t, sel] / s[t, sel].sum(), rtol=0, atol=1e-15)


def test_corr_bias_forces_and_forbids_experts():
    rng = np.random.default_rng(43)
    s = rng.random((30, 8))
    cfg = O.OracleConfig(T=30, D=1, F=1, E=8, k=2)
    b = np.zeros(8)
    b[5] = 10.0            # always chosen, first
    b[2] = -10.0           # never chosen
    idx = O.route(cfg, s, b)
    assert np.all(idx[:, 0] == 5) and not np.any(idx == 2)
    # the second choice is the best unbiased score among the rest
    rest = [e for e in range(8) if e not in (2, 5)]
    np.testing.assert_array_equal(idx[:, 1], np.array(rest)[np.argmax(s[:, rest], axis=1)])
    g = O.renormalize(s, idx)
    np.testing.assert_allclose(g[:, 0], s[:, 5] / (s[:, 5] + s[np.arange(30), idx[:, 1]]))


def test_grouped_corr_bias_brute_force():
    rng = np.random.default_rng(44)
    E, G, kg, k = 8, 4, 2, 3
    cfg = O.OracleConfig(T=60, D=1, F=1, E=E, k=k, n_groups=G, topk_groups=kg)
    s = rng.integers(0, 4, size=(60, E)).astype(np.float64) / 4.0
    b = np.array([0.0, 0.5, 0.25, -0.25, 0.0, 0.0, 0.75, -0.5])
    idx = O.route(cfg, s, b)
    for t in range(60):
        key = s[t] + b
        assert set(idx[t].tolist()) == _brute_grouped(key, k, G, kg, "top2_sum")


def test_corr_bias_keys_summed_in_float32():
    # 0.1f + 0.2f rounds to 0.3f in float32 (a tie: the smaller id wins), while
    # in float64 it stays below 0.3f (expert 1 wins)
    s32 = np.array([[0.1, 0.3]], dtype=np.float32)
    b = np.array([0.2, 0.0], dtype=np.float32)
    cfg = O.OracleConfig(T=1, D=1, F=1, E=2, k=1)
    assert O.route(cfg, s32, b).tolist() == [[0]]
    assert O.route(cfg, s32.astype(np.float64), b.astype(np.float64)).tolist() == [[1]]


@pytest.mark.parametrize("case", [dict(act="relu", score="softmax", has_bias=True, aux_alpha=0.1),
                                  dict(act="swiglu", score="sigmoid", has_bias=False, aux_alpha=0.05,
                                       E=8, n_groups=4, topk_groups=2)])
def test_corr_bias_gradients_central_differences(case):
    """With a bias that changes the routing, the oracle's analytic gradients
    still match central differences of its own loss (routing held by a margin
    on the biased keys)."""
    c = dict(T=8, D=4, F=6, E=4, k=2)
    c.update(case)
    cfg = O.OracleConfig(**c)
    found = None
    for seed in range(500, 900):
        w, x, tgt = _weights(cfg, seed, scale=1.5)
        w["corr_bias"] = np.random.default_rng(seed + 7).uniform(-0.3, 0.3, cfg.E)
        st = O.forward(cfg, w, x)
        keys = O.selection_keys(st["scores"], w["corr_bias"])
        if not np.array_equal(st["idx"], O.route(cfg, st["scores"])) and \
                np.min(np.abs(np.diff(np.sort(keys, axis=1), axis=1))) > 1e-3 and \
                (cfg.n_groups == 1 or np.min(np.abs(np.diff(np.sort(
                    O.group_scores(keys, cfg.n_groups), axis=1), axis=1))) > 1e-3) and \
                all(np.min(np.abs(fe[kk])) > 1e-3 for fe in st["experts"] for kk in ("h", "h1")
                    if kk in fe and fe[kk].size):
            found = (w, x, tgt, st)
            break
    assert found is not None
    w, x, tgt, st = found
    _, _, dy = O.losses(cfg, st, tgt)
    g = O.backward(cfg, w, x, st, dy)
    h = 1e-6
    for key in ("w_gate", "w1"):
        fd = np.zeros_like(w[key])
        for i in np.ndindex(w[key].shape):
            wp = dict(w); wp[key] = w[key].copy(); wp[key][i] += h
            wm = dict(w); wm[key] = w[key].copy(); wm[key][i] -= h
            fd[i] = (O.total_loss(cfg, wp, x, tgt) - O.total_loss(cfg, wm, x, tgt)) / (2 * h)
        err = np.max(np.abs(fd - g["d" + key])) / np.max(np.abs(fd))
        assert err <= 1e-6, (key, err)


# ----------------------------------------------------------- shared experts ---
# "AI Infra Kernel Lab": the shared branch is one SwiGLU of hidden width
# n_shared x F that every token passes through, added without a gate.

def _shared_case(seed, n_shared=2, case=None):
    c = dict(T=8, D=4, F=6, E=4, k=2, act="swiglu", score="softmax", has_bias=False,
             aux_alpha=0.01)
    if case:
        c.update(case)
    cfg = O.OracleConfig(**c)
    for s in range(seed, seed + 400):
        w, x, tgt = _weights(cfg, s, scale=1.5)
        if not _margin_ok(cfg, w, x):
            continue
        rng = np.random.default_rng(s + 1000)
        Fs = n_shared * cfg.F
        w["ws1"] = rng.normal(size=(Fs, cfg.D)) / math.sqrt(cfg.D)
        w["ws3"] = rng.normal(size=(Fs, cfg.D)) / math.sqrt(cfg.D)
        w["ws2"] = rng.normal(size=(cfg.D, Fs)) / math.sqrt(Fs)
        h1 = x @ w["ws1"].T
        if np.min(np.abs(h1)) > 1e-3:
            return cfg, w, x, tgt
    raise RuntimeError("no input found")


def test_shared_branch_vs_dense_autograd():
    cfg, w, x, tgt = _shared_case(700)
    st = O.forward(cfg, w, x)
    _, _, dy = O.losses(cfg, st, tgt)
    g = O.backward(cfg, w, x, st, dy)
    tw = {k_: torch.from_numpy(v.copy()).requires_grad_(True)
          for k_, v in w.items() if isinstance(v, np.ndarray)}
    xt = torch.from_numpy(x.copy()).requires_grad_(True)
    mask = torch.zeros(cfg.T, cfg.E, dtype=torch.float64)
    for t in range(cfg.T):
        mask[t, st["idx"][t]] = 1.0
    p = torch.softmax(xt @ tw["w_gate"].T, 1)
    gate = mask * p / (mask * p).sum(1, keepdim=True)
    F_ = torch.nn.functional
    y = F_.linear(F_.silu(F_.linear(xt, tw["ws1"])) * F_.linear(xt, tw["ws3"]), tw["ws2"])
    for e in range(cfg.E):
        hh = F_.silu(xt @ tw["w1"][e].T) * (xt @ tw["w3"][e].T)
        y = y + gate[:, e:e + 1] * (hh @ tw["w2"][e].T)
    np.testing.assert_allclose(st["y"], y.detach().numpy(), rtol=1e-12, atol=1e-14)
    mse = ((y - torch.from_numpy(tgt)) ** 2).mean()
    counts = torch.from_numpy(st["counts"].astype(np.float64))
    aux = cfg.E * (counts / (cfg.T * cfg.k) * p.mean(0)).sum()
    (mse + cfg.aux_alpha * aux).backward()
    for key in tw:
        np.testing.assert_allclose(g["d" + key], tw[key].grad.numpy(), rtol=1e-10,
                                   atol=1e-13, err_msg=key)
    np.testing.assert_allclose(g["dx"], xt.grad.numpy(), rtol=1e-10, atol=1e-13)


@pytest.mark.parametrize("case", [None, dict(score="sigmoid", E=8, n_groups=4, topk_groups=2,
                                             aux_alpha=0.0)])
def test_shared_gradients_central_differences(case):
    cfg, w, x, tgt = _shared_case(800, n_shared=1, case=case)
    st = O.forward(cfg, w, x)
    _, _, dy = O.losses(cfg, st, tgt)
    g = O.backward(cfg, w, x, st, dy)
    h = 1e-6
    for key in ("ws1", "ws3", "ws2"):
        fd = np.zeros_like(w[key])
        for i in np.ndindex(w[key].shape):
            wp = dict(w); wp[key] = w[key].copy(); wp[key][i] += h
            wm = dict(w); wm[key] = w[key].copy(); wm[key][i] -= h
            fd[i] = (O.total_loss(cfg, wp, x, tgt) - O.total_loss(cfg, wm, x, tgt)) / (2 * h)
        err = np.max(np.abs(fd - g["d" + key])) / np.max(np.abs(fd))
        assert err <= 1e-6, (key, err)
    fd = np.zeros_like(x)
    for i in np.ndindex(x.shape):
        xp = x.copy(); xp[i] += h
        xm = x.copy(); xm[i] -= h
        fd[i] = (O.total_loss(cfg, w, xp, tgt) - O.total_loss(cfg, w, xm, tgt)) / (2 * h)
    assert np.max(np.abs(fd - g["dx"])) / np.max(np.abs(fd)) <= 1e-6


def test_shared_zero_down_projection_is_identity():
    cfg, w, x, tgt = _shared_case(900)
    w0 = {k_: v for k_, v in w.items() if not k_.startswith("ws")}
    w["ws2"] = np.zeros_like(w["ws2"])
    st, st0 = O.forward(cfg, w, x), O.forward(cfg, w0, x)
    np.testing.assert_array_equal(st["y"], st0["y"])
    _, _, dy = O.losses(cfg, st, tgt)
    g = O.backward(cfg, w, x, st, dy)
    g0 = O.backward(cfg, w0, x, st0, dy)
    assert not np.any(g["dws1"]) and not np.any(g["dws3"])
    np.testing.assert_array_equal(g["dx"], g0["dx"])
    a = O.silu(x @ w["ws1"].T) * (x @ w["ws3"].T)
    np.testing.assert_allclose(g["dws2"], dy.T @ a, rtol=1e-12)


# ----------------------------------------------------- capacity / dropping ---
# Reading of the capacity factor ("AI Infra Kernel Lab" names it for dropping
# or padding tokens): C = ceil(cf T k / E); an expert keeps its first C assignments
# in token order, the rest contribute nothing and get no gradient.

def test_capacity_formula_and_no_drop_limit():
    cfg = O.OracleConfig(T=10, D=1, F=1, E=4, k=2, capacity_factor=1.25)
    assert O.expert_capacity(cfg) == 7                      # ceil(1.25 * 20 / 4) = ceil(6.25)
    assert O.expert_capacity(O.OracleConfig(T=10, D=1, F=1, E=4, k=2)) is None
    rng = np.random.default_rng(51)
    idx = np.stack([rng.permutation(6)[:3] for _ in range(40)]).astype(np.int32)
    plain = O.dispatch(idx, 6)
    big = O.dispatch(idx, 6, capacity=int(plain[0].max()))  # nothing above the cap
    for a, b in zip(plain, big):
        np.testing.assert_array_equal(a, b)


def test_capacity_dispatch_brute_force():
    rng = np.random.default_rng(52)
    T, E, k, C = 30, 5, 2, 4
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    counts, offsets, src_tok, src_j, slot_of = O.dispatch(idx, E, capacity=C)
    for e in range(E):
        order = [(t, j) for t in range(T) for j in range(k) if idx[t, j] == e]
        assert counts[e] == len(order)
        kept = order[:C]
        assert offsets[e + 1] - offsets[e] == len(kept)
        for r, (t, j) in enumerate(kept):
            s = offsets[e] + r
            assert slot_of[t, j] == s and src_tok[s] == t and src_j[s] == j
        for (t, j) in order[C:]:
            assert slot_of[t, j] == -1
    assert len(src_tok) == offsets[E] == sum(min(c, C) for c in counts)


def _capacity_case(seed):
    cfg = O.OracleConfig(T=12, D=4, F=6, E=4, k=2, act="gelu_tanh", score="softmax",
                         has_bias=True, aux_alpha=0.05, capacity_factor=0.5)
    for s in range(seed, seed + 400):
        w, x, tgt = _weights(cfg, s, scale=1.5)
        if _margin_ok(cfg, w, x):
            st = O.forward(cfg, w, x)
            if np.any(st["slot_of"] < 0) and np.any(np.all(st["slot_of"] < 0, axis=1)):
                return cfg, w, x, tgt, st
    raise RuntimeError("no input with drops found")


def test_capacity_forward_by_hand_and_zero_gate_gradients():
    cfg, w, x, tgt, st = _capacity_case(1100)
    assert O.expert_capacity(cfg) == 3
    for t in range(cfg.T):
        y = np.zeros(cfg.D)
        for j in range(cfg.k):
            if st["slot_of"][t, j] < 0:
                continue
            e = st["idx"][t, j]
            h = x[t] @ w["w1"][e].T + w["b1"][e]
            a = 0.5 * h * (1 + np.tanh(math.sqrt(2 / math.pi) * (h + 0.044715 * h ** 3)))
            y += st["gate"][t, j] * (a @ w["w2"][e].T + w["b2"][e])
        if np.all(st["slot_of"][t] < 0):
            assert not np.any(st["y"][t])                   # fully dropped: exactly 0
        np.testing.assert_allclose(st["y"][t], y, rtol=1e-12, atol=1e-15)
    _, _, dy = O.losses(cfg, st, tgt)
    g = O.backward(cfg, w, x, st, dy)
    assert np.all(g["dgate"][st["slot_of"] < 0] == 0)
    # the aux loss counts the router's assignments before any drop
    aux, f, _ = O.aux_loss(st["counts"], st["scores"], cfg.k)
    assert st["counts"].sum() == cfg.T * cfg.k and st["offsets"][-1] < cfg.T * cfg.k


def test_capacity_gradients_central_differences():
    cfg, w, x, tgt, st = _capacity_case(1200)
    _, _, dy = O.losses(cfg, st, tgt)
    g = O.backward(cfg, w, x, st, dy)
    h = 1e-6
    for key in ("w_gate", "w1", "b2"):
        fd = np.zeros_like(w[key])
        for i in np.ndindex(w[key].shape):
            wp = dict(w); wp[key] = w[key].copy(); wp[key][i] += h
            wm = dict(w); wm[key] = w[key].copy(); wm[key][i] -= h
            fd[i] = (O.total_loss(cfg, wp, x, tgt) - O.total_loss(cfg, wm, x, tgt)) / (2 * h)
        err = np.max(np.abs(fd - g["d" + key])) / np.max(np.abs(fd))
        assert err <= 1e-6, (key, err)
    fd = np.zeros_like(x)
    for i in np.ndindex(x.shape):
        xp = x.copy(); xp[i] += h
        xm = x.copy(); xm[i] -= h
        fd[i] = (O.total_loss(cfg, w, xp, tgt) - O.total_loss(cfg, w, xm, tgt)) / (2 * h)
    assert np.max(np.abs(fd - g["dx"])) / np.max(np.abs(fd)) <= 1e-6


# -------------------------------------------------------- hand-worked case ---

def _golden(name):
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", name)
    out = {}
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, rest = line.split(None, 1)
        out[key] = [[float(v) for v in part.split()] for part in rest.split("|")]
    return out


def test_hand_worked_router_dispatch_aux():
    g = _golden("hand_worked_router_dispatch.txt")
    m = np.array(g["multipliers"])
    logits = np.log(m)
    cfg = O.OracleConfig(T=3, D=1, F=1, E=4, k=2)
    p = O.softmax_rows(logits)
    np.testing.assert_allclose(p, np.array(g["scores"]), rtol=0, atol=1e-15)
    idx = O.route(cfg, p)
    np.testing.assert_array_equal(idx, np.array(g["idx"]).astype(int))
    gate = O.renormalize(p, idx)
    want = np.array(g["gate_num"]) / np.array(g["gate_den"])
    np.testing.assert_allclose(gate, want, rtol=0, atol=1e-15)
    counts, offsets, src_tok, _, slot_of = O.dispatch(idx, 4)
    np.testing.assert_array_equal(counts, np.array(g["counts"][0]).astype(int))
    np.testing.assert_array_equal(offsets, np.array(g["offsets"][0]).astype(int))
    np.testing.assert_array_equal(src_tok, np.array(g["src_tok"][0]).astype(int))
    np.testing.assert_array_equal(slot_of, np.array(g["slot_of"]).astype(int))
    aux, _, _ = O.aux_loss(counts, p, 2)
    assert abs(aux - g["aux_num"][0][0] / g["aux_den"][0][0]) <= 1e-15


def test_hand_worked_grouped_router():
    """The group-limited router on a hand-derived case: group scores by top-2
    sums (not whole-group sums), group ties to the smaller group id, expert
    ties to the smaller id, renormalised sigmoid gates, stable dispatch and
    the aux value 53/16."""
    g = _golden("hand_worked_grouped_router.txt")
    m = np.array(g["m"])
    s = m / 32.0
    cfg = O.OracleConfig(T=3, D=1, F=1, E=9, k=3, score="sigmoid", n_groups=3, topk_groups=2,
                         group_score="top2_sum")
    # the logits ln(m / (32 - m)) give the scores back through the sigmoid
    np.testing.assert_allclose(O.router_scores(cfg, np.log(m / (32.0 - m))), s,
                               rtol=0, atol=1e-15)
    idx = O.route(cfg, s)
    np.testing.assert_array_equal(idx, np.array(g["idx"]).astype(int))
    gate = O.renormalize(s, idx)
    want = np.array(g["gate_num"]) / np.array(g["gate_den"])
    np.testing.assert_allclose(gate, want, rtol=0, atol=1e-15)
    counts, offsets, src_tok, _, slot_of = O.dispatch(idx, 9)
    np.testing.assert_array_equal(counts, np.array(g["counts"][0]).astype(int))
    np.testing.assert_array_equal(offsets, np.array(g["offsets"][0]).astype(int))
    np.testing.assert_array_equal(src_tok, np.array(g["src_tok"][0]).astype(int))
    np.testing.assert_array_equal(slot_of, np.array(g["slot_of"]).astype(int))
    aux, _, _ = O.aux_loss(counts, s, 3)
    assert abs(aux - g["aux_num"][0][0] / g["aux_den"][0][0]) <= 1e-15


def test_hand_worked_expert_mlp():
    """One token through one ReLU expert with biases, every value by hand."""
    g = _golden("hand_worked_expert_mlp.txt")
    arr = lambda key: np.array(g[key])  # noqa: E731
    cfg = O.OracleConfig(T=1, D=2, F=2, E=1, k=1, act="relu", score="softmax",
                         has_bias=True, aux_alpha=0.0)
    w = dict(w_gate=np.zeros((1, 2)), w1=arr("w1")[None], w2=arr("w2")[None],
             b1=arr("b1"), b2=arr("b2"))
    x = arr("x")
    st = O.forward(cfg, w, x)
    np.testing.assert_array_equal(st["experts"][0]["h"], arr("h"))
    np.testing.assert_array_equal(st["y"], arr("y"))
    l_mse, aux, dy = O.losses(cfg, st, arr("target"))
    assert l_mse == g["mse"][0][0] and aux == g["aux"][0][0]
    gr = O.backward(cfg, w, x, st, dy)
    np.testing.assert_array_equal(gr["dw2"][0], arr("dw2"))
    np.testing.assert_array_equal(gr["db2"][0], arr("db2")[0])
    np.testing.assert_array_equal(gr["dw1"][0], arr("dw1"))
    np.testing.assert_array_equal(gr["db1"][0], arr("db1")[0])
    np.testing.assert_array_equal(gr["dx"], arr("dx"))
