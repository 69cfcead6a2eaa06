"""Parity at the full sizes of the SwiGLU layers, in the launch configuration
bench.py times (whole layer, all tokens, one training step through the C ABI).

The oracle cannot run a whole step at these sizes, so it checks what it can
compute exactly or one token at a time:
  * routing over ALL tokens, bit-exact given the GPU's own fp32 scores;
  * the scores and the aux loss against the oracle's fp64 router (cheap);
  * y, dX and the router gradient dlogits on sampled tokens, each token's k
    expert rows run by the oracle;
  * the weight gradients and SGD step of the smallest, median and largest
    non-empty experts when the oracle can afford every token routed to them
    (about 2e12 float64 flops each: all three at the large layer, the median
    one at the skewed layer, whose hot experts hold ~35k rows), and exact
    zeros for experts with no rows;
  * every bf16 working copy equal to the bf16 rounding of its updated master.
Two reductions over all tokens need the whole forward, which the oracle cannot
afford at these sizes; they are checked for consistency with what the GPU
produced: the MSE against the mean of (y - target)^2 of the GPU's own y, and
dW_g against the GPU's (sample-checked) dlogits times x in float64.  Their
oracle values are compared in full at the same layer widths on fewer tokens
(tests/test_gpu_large_shape.py and the reduced-token cases).
Expert weights are pulled to float64 one expert at a time.
"""

import numpy as np
import pytest
import torch

import workloads as W
from oracle import moe_oracle as O
from sparse_mixture_experts_softmax_gb300 import binding as B
from tests.moe_cases import (assert_close, check_routing_exact, make_layer, np64, oracle_config,
                             validated_routing)

pytestmark = pytest.mark.gpu
TOL = 2e-2


class LazyExperts:
    """[E, ...] device tensor seen as float64 experts fetched on demand; only
    the two most recently used experts stay cached (the large layer's 128
    experts would take 25 GB of host memory in float64)."""

    def __init__(self, t, keep=2):
        self.t = t
        self.keep = keep
        self.cache = {}

    def __getitem__(self, e):
        e = int(e)
        if e in self.cache:
            self.cache[e] = self.cache.pop(e)       # most recent last
        else:
            if len(self.cache) >= self.keep:
                self.cache.pop(next(iter(self.cache)))
            self.cache[e] = self.t[e].float().cpu().numpy().astype(np.float64)
        return self.cache[e]


def _oracle_weights(inp, lb):
    return dict(w_gate=np64(inp["w_gate"].to(torch.bfloat16)), w1=LazyExperts(inp["w1_bf16"]),
                corr_bias=np64(inp.get("corr_bias")),
                ws1=np64(inp.get("ws1_bf16")), ws3=np64(inp.get("ws3_bf16")),
                ws2=np64(inp.get("ws2_bf16")),
                w2=LazyExperts(inp["w2_bf16"]),
                w3=LazyExperts(inp["w3_bf16"]) if inp["w3_bf16"] is not None else None,
                b1=None, b2=None, logit_bias=lb)


def _rows_forward(cfg, w, x64, pairs):
    """Expert rows (t, e) through the oracle's expert MLP, batched per expert.
    Returns {(t, e): forward dict of that single row}."""
    out = {}
    by_e = {}
    for t, e in pairs:
        by_e.setdefault(int(e), []).append(int(t))
    for e, ts in by_e.items():
        fe = O.expert_forward(cfg, e, x64[ts], w)
        for i, t in enumerate(ts):
            out[(t, e)] = {k_: v[i:i + 1] for k_, v in fe.items()}
    return out


def _tokens_y(cfg, w, x64, scores64, idx, tokens, kept=None):
    """y[t] for the given tokens (oracle gates from its own scores), with the
    shared-expert branch when the layer has one; ``kept[t, j]`` False marks an
    assignment dropped by the expert capacity (no output)."""
    if kept is None:
        kept = np.ones(idx.shape, dtype=bool)
    pairs = [(t, idx[t, j]) for t in tokens for j in range(cfg.k) if kept[t, j]]
    fw = _rows_forward(cfg, w, x64, pairs)
    gate = O.renormalize(scores64[tokens], idx[tokens])
    sh = O.shared_forward(x64[tokens], w) if w.get("ws1") is not None else None
    ys = {}
    for i, t in enumerate(tokens):
        y = np.zeros(cfg.D)
        for j in range(cfg.k):
            if kept[t, j]:
                y = y + gate[i, j] * fw[(t, int(idx[t, j]))]["ye"][0]
        if sh is not None:
            y = y + sh["ys"][i]
        ys[t] = y
    return ys, fw, gate


def _expert_rows_dw(cfg, w, x64, scores64, idx, kept, target, e_sel, rows_tok, T, D):
    """dW1 / dW3 / dW2 of expert ``e_sel`` from the oracle, over the tokens
    ``rows_tok`` routed to it.  Each token's y runs through all of its k
    experts first (for dY), streamed one expert at a time so that only that
    expert's float64 weights and outputs are held."""
    n = len(rows_tok)
    pos = {t: i for i, t in enumerate(rows_tok)}
    gate = O.renormalize(scores64[rows_tok], idx[rows_tok])
    y = np.zeros((n, D))
    by_e = {}
    for i, t in enumerate(rows_tok):
        for j in range(cfg.k):
            if kept[t, j]:
                by_e.setdefault(int(idx[t, j]), []).append((i, j))
    for e in sorted(by_e):
        ij = by_e[e]
        ts = [rows_tok[i] for i, _ in ij]
        ye = O.expert_forward(cfg, e, x64[ts], w)["ye"]
        for r, (i, j) in enumerate(ij):
            y[i] += gate[i, j] * ye[r]
    if w.get("ws1") is not None:
        y += O.shared_forward(x64[rows_tok], w)["ys"]
    dye = np.zeros((n, D))
    for i, t in enumerate(rows_tok):
        j = int(np.nonzero(idx[t] == e_sel)[0][0])
        assert kept[t, j]
        dye[i] = gate[i, j] * 2.0 * (y[i] - target[pos[t]]) / float(T * D)
    xe = x64[rows_tok]
    fe = O.expert_forward(cfg, e_sel, xe, w)
    return O.expert_backward(cfg, e_sel, xe, fe, dye, w)


def _run_full(name):
    wl = W.WORKLOADS[name]
    inp = W.make_inputs(wl, seed=0, device="cuda")
    cfg = oracle_config(wl)
    layer = make_layer(wl, inp)
    x = inp["x_bf16"]
    tgt = inp["target"]
    y = layer.forward(x).clone()
    dx = torch.empty(wl.T, wl.D, device="cuda")
    layer.train_step(x, tgt, wl.lr, dx=dx)
    dlogits = torch.empty(wl.T, wl.E, device="cuda")
    B.moe_get_intermediates(layer.cfg, layer.workspace, dlogits=dlogits)
    torch.cuda.synchronize()
    r = layer.routing()
    r["dlogits"] = dlogits
    return wl, inp, cfg, layer, y, dx, r


@pytest.mark.parametrize("name,n_sample", [("grouped", 8), ("skewed", 6), ("large", 4),
                                           ("grouped_cb", 8), ("grouped_shared", 8),
                                           ("skewed_cap", 12)])
def test_full_size_layer(name, n_sample):
    wl, inp, cfg, layer, y, dx, r = _run_full(name)
    T, D, E, k = wl.T, wl.D, wl.E, wl.k
    # 1. routing over all tokens, bit-exact given the GPU's scores
    check_routing_exact(cfg, r, inp.get("corr_bias"))
    idx = r["idx"].cpu().numpy()
    counts = r["counts"].cpu().numpy().astype(np.int64)
    offsets = r["offsets"].cpu().numpy()
    src_tok = r["src_tok"].cpu().numpy()
    kept = r["slot_of"].cpu().numpy() >= 0     # checked against the oracle's dispatch above
    # 2. scores and aux against the oracle's fp64 router on all tokens
    lb = np64(inp["logit_bias"])
    w = _oracle_weights(inp, lb)
    x64 = np64(inp["x_bf16"])
    scores64 = O.router_scores(cfg, O.router_logits(x64, w["w_gate"], lb))
    assert_close("scores", r["scores"].cpu().numpy(), scores64, 1e-4)
    aux, f, _ = O.aux_loss(counts, scores64, k)
    loss = layer.d_loss.cpu().numpy()
    assert_close("aux", loss[1], aux, 1e-4)
    # 3. the MSE reduction against the GPU's own y
    y64 = y.double()
    mse_of_y = float(((y64 - inp["target"].double()) ** 2).mean())
    assert_close("mse", loss[0], mse_of_y, 1e-4)
    # 4. sampled tokens: y and dX
    tokens = W.sample_tokens(T, n_sample).tolist()
    cb64 = np64(inp.get("corr_bias"))
    idx_v = validated_routing(cfg, scores64[tokens], idx[tokens], corr_bias=cb64)
    idx_s = idx.copy()
    idx_s[tokens] = idx_v
    ys, fw, gate = _tokens_y(cfg, w, x64, scores64, idx_s, tokens, kept)
    t64 = inp["target"][tokens].double().cpu().numpy()
    aux_row = cfg.aux_alpha * O.aux_loss_score_grad(counts / float(T * k), T)
    for i, t in enumerate(tokens):
        assert_close(f"y[{t}]", y[t].double().cpu().numpy(), ys[t], TOL)
        dy = 2.0 * (ys[t] - t64[i]) / float(T * D)
        dxt = np.zeros(D)
        dgate = np.zeros(k)
        for j in range(k):
            if not kept[t, j]:
                continue
            e = int(idx_s[t, j])
            fe = fw[(t, e)]
            be = O.expert_backward(cfg, e, x64[t:t + 1], fe, (gate[i, j] * dy)[None], w)
            dxt = dxt + be["dxe"][0]
            dgate[j] = float(np.dot(dy, fe["ye"][0]))
        if w.get("ws1") is not None:
            dxt = dxt + O.shared_backward(x64[t:t + 1], O.shared_forward(x64[t:t + 1], w),
                                          dy[None], w)["dx"][0]
        ds = O.renormalize_backward(scores64[t:t + 1], idx_s[t:t + 1], gate[i:i + 1], dgate[None])
        ds = ds + aux_row[None, :]
        if cfg.score == "softmax":
            dl = O.softmax_rows_backward(scores64[t:t + 1], ds)
        else:
            dl = O.sigmoid_backward(scores64[t:t + 1], ds)
        dxt = dxt + (dl @ w["w_gate"])[0]
        assert_close(f"dlogits[{t}]", r["dlogits"][t].double().cpu().numpy(), dl[0], TOL)
        assert_close(f"dx[{t}]", dx[t].double().cpu().numpy(), dxt, TOL)
    # dW_g in full: the GPU's dlogits (checked on the samples above) times x,
    # summed in float64, must give the GPU's router weight gradient
    dwg_want = (r["dlogits"].double().T @ inp["x_bf16"].double()).cpu().numpy()
    assert_close("dW_g", np64(layer.dw_gate), dwg_want, TOL)
    # 5. empty experts: exact zero gradients
    for e in np.nonzero(counts == 0)[0]:
        assert torch.all(layer.dw1[e] == 0) and torch.all(layer.dw2[e] == 0)
        assert torch.all(layer.dw3[e] == 0)
    # 6. weight gradients and SGD step of the smallest, median and largest
    #    non-empty experts, each when the oracle can afford all its tokens
    rows_kept = np.diff(offsets)              # rows each expert processed (after any drop)
    nonzero = np.nonzero(rows_kept)[0]
    order = nonzero[np.argsort(rows_kept[nonzero], kind="stable")]
    picks = []
    for e_sel in (order[0], order[len(order) // 2], order[-1]):
        if int(e_sel) not in picks:
            picks.append(int(e_sel))
    report = []
    for e_min in picks:
        n_rows = int(rows_kept[e_min])
        # oracle cost: every routed row of those tokens forward, one expert backward
        checked_dw = n_rows * k * 6 * D * wl.F <= 2e12
        report.append(f"expert {e_min} ({n_rows} rows) {'checked' if checked_dw else 'skipped'}")
        if not checked_dw:
            continue
        rows_tok = src_tok[offsets[e_min]:offsets[e_min + 1]].tolist()
        idx_v = validated_routing(cfg, scores64[rows_tok], idx[rows_tok], corr_bias=cb64)
        idx_m = idx.copy()
        idx_m[rows_tok] = idx_v
        t_rows = inp["target"][rows_tok].double().cpu().numpy()
        be = _expert_rows_dw(cfg, w, x64, scores64, idx_m, kept, t_rows, e_min, rows_tok, T, D)
        for key in ("w1", "w3", "w2"):
            assert_close(f"d{key}[{e_min}]", np64(getattr(layer, "d" + key)[e_min]), be["d" + key],
                         TOL)
            # the SGD step of that expert: theta_1 - theta_0 against -lr * grad
            # (tolerance widened by half an fp32 ulp of |theta|)
            w0 = np64(inp[key][e_min])
            step = np64(getattr(layer, key)[e_min]) - w0
            want = -wl.lr * be["d" + key]
            scale = np.max(np.abs(want))
            assert_close(f"step {key}[{e_min}]", step, want,
                         TOL + 2.0 ** -24 * np.max(np.abs(w0)) / scale)
    print(f"\n{name}: T={T} R={T * k} routed rows checked bit-exact; sampled tokens {tokens}; "
          f"{int((counts == 0).sum())} empty experts; dW of " + ", ".join(report))
    # 7. every expert's bf16 working copy is the round-to-nearest image of its
    #    updated fp32 master
    for key in ("w1", "w3", "w2") + (("ws1", "ws3", "ws2") if wl.n_shared else ()):
        assert torch.equal(getattr(layer, key + "_lp"), getattr(layer, key).to(torch.bfloat16)), key
    del layer, inp
    torch.cuda.empty_cache()
