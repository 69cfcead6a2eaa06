"""Parity of the CUDA library (through its C ABI) with the float64 oracle.

Routing is bit-exact given the GPU's own fp32 scores; float results meet the
max-norm relative tolerance 1e-4 (fp32 layers) or 2e-2 (bf16 layers), on
outputs, losses, every gradient and the updated weights.
"""

import numpy as np
import pytest
import torch

import workloads as W
from oracle import moe_oracle as O
from tests.moe_cases import (TOL, assert_close, check_routing_exact, device_x, make_layer, np64,
                             oracle_config, oracle_inputs, rel_err, validated_relu_decisions,
                             validated_routing)

pytestmark = pytest.mark.gpu


def _grad_keys(wl):
    keys = ["dw_gate", "dw1", "dw2"]
    if wl.act == "swiglu":
        keys.append("dw3")
    if wl.has_bias:
        keys += ["db1", "db2"]
    if wl.n_shared:
        keys += ["dws1", "dws3", "dws2"]
    return keys


def _one_step_parity(wl, seed=0, check_dx=True, keep=None):
    """One training step on both sides; returns the errors by tensor.  When
    ``keep`` is a dict it receives the oracle's forward state ``st``, its
    gradients ``g``, the fp32 masters before the step ``master``, the
    forward weights ``w_fwd`` and ``x64``, the output ``y`` of a forward call
    made before the step and the step's ``dx``, for further checks by the
    caller."""
    inp = W.make_inputs(wl, seed=seed)
    cfg = oracle_config(wl)
    tol = TOL[wl.dtype]
    layer = make_layer(wl, inp)
    x = device_x(wl, inp)
    tgt = inp["target"].cuda()
    dx = torch.empty(wl.T, wl.D, device="cuda")
    y_fwd = layer.forward(x).clone() if keep is not None else None   # forward alone, before the step
    layer.train_step(x, tgt, wl.lr, dx=dx)
    torch.cuda.synchronize()
    r = layer.routing()
    check_routing_exact(cfg, r, inp.get("corr_bias"))

    w_fwd, master, x64, t64 = oracle_inputs(wl, inp)
    # the oracle's own fp64 scores (the first steps of its forward) decide
    # which GPU routing decisions are near-ties to take from the kernel
    scores64 = O.router_scores(cfg, O.router_logits(x64, w_fwd["w_gate"], w_fwd.get("logit_bias")))
    idx = validated_routing(cfg, scores64, r["idx"].cpu().numpy(),
                            corr_bias=w_fwd.get("corr_bias"))
    st = O.forward(cfg, w_fwd, x64, idx)
    if wl.act == "relu":
        # kept rows only: rows past the last kept row of a capacity are unspecified
        h_kept = layer.hidden()["h1"][: int(r["offsets"][-1].item())]
        validated_relu_decisions(cfg, st, w_fwd, np64(h_kept))
    l_mse, aux, dy = O.losses(cfg, st, t64)
    g = O.backward(cfg, w_fwd, x64, st, dy)
    errs = {}
    loss = layer.d_loss.cpu().numpy()
    errs["mse"] = assert_close("mse", loss[0], l_mse, tol)
    errs["aux"] = assert_close("aux", loss[1], aux, tol)
    got = layer.grad_dict()
    for key in _grad_keys(wl):
        errs[key] = assert_close(key, np64(got[key]), g[key], tol)
    if check_dx:
        errs["dx"] = assert_close("dx", np64(dx), g["dx"], tol)
    # SGD: theta_1 = theta_0 - lr * grad on the fp32 masters
    new = layer.param_dict()
    for key in ("w_gate", "w1", "w2", "w3", "b1", "b2", "ws1", "ws3", "ws2"):
        if master.get(key) is None:
            continue
        want = master[key] - wl.lr * g["d" + key]
        errs[key] = assert_close(key, np64(new[key]), want, tol)
        # the update itself: lr * grad is far below |theta|, so compare the
        # step theta_1 - theta_0 with -lr * grad; storing theta_1 in fp32
        # adds up to half an ulp of |theta| to it
        step = np64(new[key]) - master[key]
        want_step = -wl.lr * g["d" + key]
        scale = np.max(np.abs(want_step))
        step_tol = tol + 2.0 ** -24 * np.max(np.abs(master[key])) / scale if scale > 0 else tol
        assert_close("step " + key, step, want_step, step_tol)
    if wl.dtype == "bf16":
        # the bf16 working copies are the round-to-nearest images of the masters
        for key in ("w1", "w2", "w3", "ws1", "ws3", "ws2"):
            lp = getattr(layer, key + "_lp")
            if lp is not None:
                assert torch.equal(lp, new[key].to(torch.bfloat16)), key
    if keep is not None:
        keep.update(st=st, g=g, master=master, w_fwd=w_fwd, x64=x64, y=y_fwd, dx=dx)
    return errs, layer, inp


def test_tiny_20_step_loop():
    """The fp32 tiny layer trained for 20 SGD steps: routing bit-exact at every
    step, losses / gradients / weights within 1e-4 at every step, and the
    accumulated weight change W_20 - W_0 within 1e-4."""
    wl = W.WORKLOADS["tiny"]
    inp = W.make_inputs(wl, seed=0)
    cfg = oracle_config(wl)
    layer = make_layer(wl, inp)
    x = device_x(wl, inp)
    tgt = inp["target"].cuda()
    w_fwd, master, x64, t64 = oracle_inputs(wl, inp)
    w0 = {k: v.copy() for k, v in master.items() if v is not None}
    wo = dict(w_fwd)
    dx = torch.empty(wl.T, wl.D, device="cuda")
    losses_gpu = []
    for step in range(wl.steps):
        layer.train_step(x, tgt, wl.lr, dx=dx)
        torch.cuda.synchronize()
        r = layer.routing()
        check_routing_exact(cfg, r)
        st0 = O.forward(cfg, wo, x64)
        idx = validated_routing(cfg, st0["scores"], r["idx"].cpu().numpy())
        wo_new, (l_mse, aux), st, g = O.train_step(cfg, wo, x64, t64, wl.lr, idx)
        loss = layer.d_loss.cpu().numpy()
        losses_gpu.append(float(loss[0] + wl.aux_alpha * loss[1]))
        assert_close(f"mse@{step}", loss[0], l_mse, 1e-4)
        assert_close(f"aux@{step}", loss[1], aux, 1e-4)
        for key in _grad_keys(wl):
            assert_close(f"{key}@{step}", np64(layer.grad_dict()[key]), g[key], 1e-4)
        assert_close(f"dx@{step}", np64(dx), g["dx"], 1e-4)
        wo = wo_new
        for key, v in layer.param_dict().items():
            if v is not None:
                assert_close(f"{key}@{step}", np64(v), wo[key], 1e-4)
    for key, v in layer.param_dict().items():
        if v is not None:
            assert_close(f"delta {key}", np64(v) - w0[key], wo[key] - w0[key], 1e-4)
    assert losses_gpu[-1] < losses_gpu[0]


def test_dense_f32_step():
    errs, _, _ = _one_step_parity(W.WORKLOADS["dense_f32"])
    assert max(errs.values()) <= 1e-4


def test_dense_bf16_step():
    errs, _, _ = _one_step_parity(W.WORKLOADS["dense_bf16"])
    assert max(errs.values()) <= 2e-2


def test_correction_bias_f32_step():
    """fp32 fused router with a selection-only correction bias: the bias moves
    routing decisions (checked), gates and all gradients from unbiased scores."""
    wl = W.WORKLOADS["dense_f32_cb"]
    errs, layer, inp = _one_step_parity(wl)
    assert max(errs.values()) <= 1e-4
    _assert_bias_changes_routing(wl, inp, layer)


def test_correction_bias_grouped_bf16_step():
    """Grouped sigmoid routing with a correction bias on the tensor-core router
    (group scores from the biased keys), at the layer's full width, 2048 tokens."""
    wl = W.WORKLOADS["grouped_cb"].with_tokens(2048)
    errs, layer, inp = _one_step_parity(wl, check_dx=True)
    assert max(errs.values()) <= 2e-2
    _assert_bias_changes_routing(wl, inp, layer)


@pytest.mark.parametrize("T", [2048, 777])
def test_shared_experts_step(T):
    """Shared-expert SwiGLU branch (width 2F, every token, no gate) on the
    grouped layer: forward through combine, its dA / dX / dW GEMMs, the scatter
    of its dX, and its fused SGD step (a ragged token count included)."""
    wl = W.WORKLOADS["grouped_shared"].with_tokens(T)
    errs, layer, _ = _one_step_parity(wl)
    assert max(errs.values()) <= 2e-2
    assert layer.dws1.abs().max().item() > 0 and layer.dws2.abs().max().item() > 0


def test_shared_experts_forward_backward_entry_points():
    """moe_forward / moe_backward (external dY, fp32) with the shared branch."""
    wl = W.WORKLOADS["grouped_shared"].with_tokens(1024)
    inp = W.make_inputs(wl, seed=5)
    cfg = oracle_config(wl)
    layer = make_layer(wl, inp)
    x = device_x(wl, inp)
    y = layer.forward(x)
    w_fwd, _, x64, t64 = oracle_inputs(wl, inp)
    st0 = O.forward(cfg, w_fwd, x64)
    idx = validated_routing(cfg, st0["scores"], layer.routing()["idx"].cpu().numpy())
    st = O.forward(cfg, w_fwd, x64, idx)
    assert_close("y", np64(y), st["y"], 2e-2)
    _, _, dy = O.losses(cfg, st, t64)
    dyt = torch.from_numpy(dy.astype(np.float32)).cuda()
    dx = torch.empty_like(dyt)
    layer.backward(x, dyt, dx)
    g = O.backward(cfg, w_fwd, x64, st, dy)
    for key in _grad_keys(wl):
        assert_close(key, np64(layer.grad_dict()[key]), g[key], 2e-2)
    assert_close("dx", np64(dx), g["dx"], 2e-2)


@pytest.mark.parametrize("name,T", [("dense_f32_cap", 4096), ("skewed_cap", 1536)])
def test_capacity_factor_step(name, T):
    """Expert capacity: each expert keeps its first C assignments in token
    order; dropped ones contribute nothing and their gates get zero gradient.
    Checks that drops occur, then full one-step parity."""
    wl = W.WORKLOADS[name].with_tokens(T)
    errs, layer, inp = _one_step_parity(wl)
    assert max(errs.values()) <= TOL[wl.dtype]
    r = layer.routing()
    dropped = int((r["slot_of"] < 0).sum().item())
    kept_rows = int(r["offsets"][-1].item())
    assert dropped > 0 and kept_rows + dropped == wl.T * wl.k


def _assert_bias_changes_routing(wl, inp, layer):
    """The bias must matter for this input: the oracle's routing of the GPU's
    scores without the bias differs on a good share of tokens."""
    cfg = oracle_config(wl)
    r = layer.routing()
    scores = r["scores"].cpu().numpy()
    plain = O.route(cfg, scores)
    changed = np.mean(np.any(plain != r["idx"].cpu().numpy(), axis=1))
    assert changed > 0.05, changed


@pytest.mark.parametrize("name,T", [("grouped", 2048), ("skewed", 768), ("large", 256)])
def test_swiglu_layers_reduced_tokens(name, T):
    """The SwiGLU layers at their full width (D, F, E, k) on fewer tokens, so
    the oracle finishes in seconds: ragged expert segments, F = 704 tails,
    empty experts (skewed), grouped sigmoid routing (grouped)."""
    wl = W.WORKLOADS[name].with_tokens(T)
    errs, layer, _ = _one_step_parity(wl)
    if name == "skewed":
        counts = layer.routing()["counts"].cpu().numpy()
        assert (counts == 0).sum() >= 4
        empty = np.nonzero(counts == 0)[0]
        for e in empty:
            assert torch.all(layer.dw1[e] == 0) and torch.all(layer.dw2[e] == 0)
            assert torch.all(layer.dw3[e] == 0)


def test_forward_backward_match_train_step():
    """moe_forward + moe_backward give the same bits as the train step's
    forward and backward; forward output y matches the oracle."""
    wl = W.WORKLOADS["dense_f32"].with_tokens(1000)
    inp = W.make_inputs(wl, seed=3)
    cfg = oracle_config(wl)
    layer = make_layer(wl, inp)
    x = device_x(wl, inp)
    y = layer.forward(x)
    w_fwd, _, x64, t64 = oracle_inputs(wl, inp)
    st0 = O.forward(cfg, w_fwd, x64)
    idx = validated_routing(cfg, st0["scores"], layer.routing()["idx"].cpu().numpy())
    st = O.forward(cfg, w_fwd, x64, idx)
    assert_close("y", np64(y), st["y"], 1e-4)
    _, _, dy = O.losses(cfg, st, t64)
    dyt = torch.from_numpy(dy.astype(np.float32)).cuda()
    dx = torch.empty_like(dyt)
    layer.backward(x, dyt, dx)
    g = O.backward(cfg, w_fwd, x64, st, dy)
    for key in _grad_keys(wl):
        assert_close(key, np64(layer.grad_dict()[key]), g[key], 1e-4)
    assert_close("dx", np64(dx), g["dx"], 1e-4)


def test_deterministic_and_inputs_unchanged():
    wl = W.WORKLOADS["dense_bf16"].with_tokens(1500)
    inp = W.make_inputs(wl, seed=5)
    layer = make_layer(wl, inp)
    x = device_x(wl, inp)
    x_copy = x.clone()
    w_copy = {k: v.clone() for k, v in layer.param_dict().items() if v is not None}
    y1 = layer.forward(x).clone()
    dy = torch.randn(wl.T, wl.D, device="cuda") * 1e-3
    dx1 = layer.backward(x, dy, torch.empty_like(dy)).clone()
    g1 = {k: v.clone() for k, v in layer.grad_dict().items() if v is not None}
    y2 = layer.forward(x)
    dx2 = layer.backward(x, dy, torch.empty_like(dy))
    assert torch.equal(y1, y2) and torch.equal(dx1, dx2)
    for k, v in layer.grad_dict().items():
        if v is not None:
            assert torch.equal(g1[k], v), k
    assert torch.equal(x, x_copy)
    for k, v in layer.param_dict().items():
        if v is not None:
            assert torch.equal(w_copy[k], v), k


def test_host_entry_point_matches_device():
    from sparse_mixture_experts_softmax_gb300 import binding as B
    wl = W.WORKLOADS["dense_f32"].with_tokens(640)
    inp = W.make_inputs(wl, seed=6)
    a = make_layer(wl, inp)
    b = make_layer(wl, inp)
    x = device_x(wl, inp)
    tgt = inp["target"].cuda()
    a.train_step(x, tgt, wl.lr)
    staging = torch.empty(B.moe_host_staging_size(b.cfg), dtype=torch.uint8, device="cuda")
    loss_host = torch.zeros(2, dtype=torch.float32).pin_memory()
    B.moe_train_step_host(b.cfg, b.params(), x.cpu().pin_memory(), inp["target"].pin_memory(),
                          wl.lr, loss_host, staging, b.workspace)
    torch.cuda.synchronize()
    assert torch.equal(a.d_loss.cpu(), loss_host)
    for k, v in a.param_dict().items():
        if v is not None:
            assert torch.equal(v, b.param_dict()[k]), k


def test_pipelined_host_steps_match_sequential_steps():
    """moe_train_steps_host over three different host batches (inputs of step
    i+1 uploaded while step i runs) gives bit-identical losses and weights to
    three moe_train_step calls in order."""
    from sparse_mixture_experts_softmax_gb300 import binding as B
    wl = W.WORKLOADS["dense_bf16"].with_tokens(777)
    batches = [W.make_inputs(wl, seed=s) for s in (21, 22, 23)]
    inp = batches[0]
    a = make_layer(wl, inp)
    b = make_layer(wl, inp)
    losses_a = []
    for bt in batches:
        a.train_step(device_x(wl, bt), bt["target"].cuda(), wl.lr)
        losses_a.append(a.d_loss.cpu().clone())
    xs = [bt["x_bf16"].contiguous().pin_memory() for bt in batches]
    ts = [bt["target"].contiguous().pin_memory() for bt in batches]
    staging = torch.empty(2 * B.moe_host_staging_size(b.cfg), dtype=torch.uint8, device="cuda")
    loss_host = torch.zeros(2 * len(batches), dtype=torch.float32).pin_memory()
    B.moe_train_steps_host(b.cfg, b.params(), xs, ts, wl.lr, loss_host, staging, b.workspace)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(losses_a), loss_host)
    for k, v in a.param_dict().items():
        if v is not None:
            assert torch.equal(v, b.param_dict()[k]), k
    for k in ("w1", "w2"):
        assert torch.equal(getattr(a, k + "_lp"), getattr(b, k + "_lp")), k


def test_host_entry_points_from_two_threads():
    """Two host threads drive moe_train_steps_host and moe_train_step_host on
    one device at once, each with its own layer, stream, staging and batches
    (the library serialises these calls per device).  Each thread's losses and
    weights are bit-identical to the same call sequence made alone."""
    import threading
    from sparse_mixture_experts_softmax_gb300 import binding as B
    wl = W.WORKLOADS["dense_bf16"].with_tokens(640)
    seeds = {0: (31, 32, 33), 1: (41, 42, 43)}
    batches = {w: [W.make_inputs(wl, seed=s) for s in seeds[w]] for w in seeds}
    host = {w: ([bt["x_bf16"].contiguous().pin_memory() for bt in batches[w]],
                [bt["target"].contiguous().pin_memory() for bt in batches[w]]) for w in seeds}

    def sequence(layer, w, stream, out):
        xs, ts = host[w]
        with torch.cuda.stream(stream):
            staging = torch.empty(2 * B.moe_host_staging_size(layer.cfg), dtype=torch.uint8,
                                  device="cuda")
            losses = torch.zeros(2 * len(xs), dtype=torch.float32).pin_memory()
            loss1 = torch.zeros(2, dtype=torch.float32).pin_memory()
            for _ in range(3):
                B.moe_train_steps_host(layer.cfg, layer.params(), xs, ts, wl.lr, losses, staging,
                                       layer.workspace, stream=stream)
                out.append(losses.clone())
                B.moe_train_step_host(layer.cfg, layer.params(), xs[1], ts[1], wl.lr, loss1,
                                      staging, layer.workspace, stream=stream)
                out.append(loss1.clone())
            stream.synchronize()

    alone, together = {}, {}
    for w in seeds:   # each sequence alone, one after the other
        layer = make_layer(wl, batches[w][0])
        torch.cuda.synchronize()   # the layer's set-up ran on the default stream
        out = []
        sequence(layer, w, torch.cuda.Stream(), out)
        alone[w] = (out, {k: v.clone() for k, v in layer.param_dict().items() if v is not None})
    layers = {w: make_layer(wl, batches[w][0]) for w in seeds}
    streams = {w: torch.cuda.Stream() for w in seeds}
    torch.cuda.synchronize()
    outs = {w: [] for w in seeds}
    errors = []

    def worker(w):
        try:
            sequence(layers[w], w, streams[w], outs[w])
        except Exception as e:   # surfaced on the main thread below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(w,)) for w in seeds]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for w in seeds:
        ref_losses, ref_params = alone[w]
        assert len(outs[w]) == len(ref_losses)
        for a, b in zip(ref_losses, outs[w]):
            assert torch.equal(a, b), w
        for k, v in layers[w].param_dict().items():
            if v is not None:
                assert torch.equal(ref_params[k], v), (w, k)


def test_all_routing_options_together():
    """Correction bias + shared experts + expert capacity on the grouped layer
    at once (full width, 1024 tokens): the options compose."""
    import dataclasses
    wl = dataclasses.replace(W.WORKLOADS["grouped"], name="grouped_all", T=1024,
                             corr_bias_scale=0.1, n_shared=1, capacity_factor=1.0)
    errs, layer, _ = _one_step_parity(wl)
    assert max(errs.values()) <= 2e-2
    assert int((layer.routing()["slot_of"] < 0).sum().item()) > 0


@pytest.mark.parametrize("name", ["dense_bf16", "dense_f32"])
def test_cuda_graph_replay_matches_eager(name):
    """After one eager call, a training step captures into a CUDA graph (no
    host synchronisation or allocation inside); three replays give the same
    bits as three eager steps (the fp32 layer with its GEMMs on the tensor
    cores through the three-term split, the operand expansion included)."""
    wl = W.WORKLOADS[name].with_tokens(1000)
    inp = W.make_inputs(wl, seed=8)
    a = make_layer(wl, inp)
    b = make_layer(wl, inp)
    x = device_x(wl, inp)
    tgt = inp["target"].cuda()
    for _ in range(4):
        a.train_step(x, tgt, wl.lr)
    b.train_step(x, tgt, wl.lr)                  # eager first call (one-time setup)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            b.train_step(x, tgt, wl.lr)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(a.d_loss, b.d_loss)
    for k, v in a.param_dict().items():
        if v is not None:
            assert torch.equal(v, b.param_dict()[k]), k


@pytest.mark.parametrize("E,k,T", [(256, 8, 1536), (64, 12, 700), (16, 16, 300)])
def test_wide_routing_bf16(E, k, T):
    """The largest expert count (256: eight score registers per lane, the
    GEMM's segment table at its limit) and k > 8 (the training step then runs
    the separate combine and combine-backward kernels) on a bf16 SwiGLU layer;
    k = E = 16 routes every token to every expert."""
    import dataclasses
    wl = dataclasses.replace(W.WORKLOADS["grouped"], name=f"wide_{E}_{k}", T=T, D=256, F=128,
                             E=E, k=k, n_groups=1, topk_groups=1, score="softmax",
                             aux_alpha=0.01)
    errs, _, _ = _one_step_parity(wl, seed=13)
    assert max(errs.values()) <= 2e-2


# tiny: CUDA-core GEMMs; the 256 x 256 fp32 layer: the tensor-core path
# through the three-term split
SPLIT_F32 = dict(D=256, F=256, act="gelu_tanh")


def test_swiglu_f32_split_step():
    """An fp32 SwiGLU layer wide enough for the tensor-core path: H1 = X W1^T,
    dXe over both pairs (dH1 W1 + dH3 W3) and the weight gradients through the
    three-term split; the W3 product with the SwiGLU epilogue and the SwiGLU
    backward on the CUDA cores."""
    import dataclasses
    wl = dataclasses.replace(W.WORKLOADS["tiny"], name="swiglu_f32_split", T=300, D=256, F=512,
                             E=8, k=2, act="swiglu", has_bias=False)
    errs, _, _ = _one_step_parity(wl, seed=17)
    assert max(errs.values()) <= 1e-4


@pytest.mark.parametrize("split", [False, True])
def test_empty_tokens(split):
    import dataclasses
    wl = W.WORKLOADS["tiny"]
    if split:
        wl = dataclasses.replace(wl, **SPLIT_F32)
    inp = W.make_inputs(wl, seed=0)
    layer = make_layer(wl.with_tokens(0), {**inp, "x": inp["x"][:0], "target": inp["target"][:0]})
    x = torch.empty(0, wl.D, device="cuda")
    layer.dw1.fill_(1.0)
    layer.train_step(x, torch.empty(0, wl.D, device="cuda"), wl.lr)
    torch.cuda.synchronize()
    assert layer.d_loss.abs().sum().item() == 0.0
    assert torch.all(layer.dw1 == 0)


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (1, 2, 4), (37, 4, 4), (130, 1, 3)])
def test_edge_shapes(T, k, E, split):
    """Single token, single expert, k = E, odd token counts; on the CUDA-core
    GEMMs and on the tensor-core path of fp32 layers."""
    base = W.WORKLOADS["tiny"]
    import dataclasses
    wl = dataclasses.replace(base, T=T, k=k, E=E, **(SPLIT_F32 if split else {}))
    errs, _, _ = _one_step_parity(wl, seed=11)
    assert max(errs.values()) <= 1e-4


@pytest.mark.parametrize("name,T", [("grouped_shared", 1000), ("dense_bf16", 900),
                                    ("dense_f32", 700)])
def test_unstored_gradients_give_identical_steps(name, T):
    """A training step whose caller passes NULL gradient buffers still applies
    every gradient: two steps give bit-identical losses, fp32 masters and bf16
    copies to the same steps with every gradient stored (bf16 layers then skip
    the expert weights' gradient store inside the fused SGD epilogue; fp32
    layers and the router / bias gradients use workspace stand-ins)."""
    from sparse_mixture_experts_softmax_gb300.layer import MoELayer as L_
    wl = W.WORKLOADS[name].with_tokens(T)
    inp = W.make_inputs(wl, seed=17)
    a = make_layer(wl, inp)
    lp = wl.dtype == "bf16"
    b = L_(wl.T, wl.D, wl.F, wl.E, wl.k, wl.act, wl.score, wl.dtype, wl.has_bias, wl.aux_alpha,
           inp["w_gate"], inp["w1"], inp["w2"], w3=inp["w3"], b1=inp["b1"], b2=inp["b2"],
           logit_bias=inp["logit_bias"], n_groups=wl.n_groups, topk_groups=wl.topk_groups,
           w1_lp=inp.get("w1_bf16") if lp else None, w3_lp=inp.get("w3_bf16") if lp else None,
           w2_lp=inp.get("w2_bf16") if lp else None, corr_bias=inp.get("corr_bias"),
           n_shared=wl.n_shared, ws1=inp.get("ws1"), ws3=inp.get("ws3"), ws2=inp.get("ws2"),
           capacity_factor=wl.capacity_factor, store_grads=False)
    assert b.dw1 is None and b.dw_gate is None
    x = device_x(wl, inp)
    tgt = inp["target"].cuda()
    for _ in range(2):
        a.train_step(x, tgt, wl.lr)
        b.train_step(x, tgt, wl.lr)
        torch.cuda.synchronize()
        assert torch.equal(a.d_loss, b.d_loss)
    for k_, v in a.param_dict().items():
        if v is not None:
            assert torch.equal(v, b.param_dict()[k_]), k_
    for k_ in ("w1", "w2", "w3", "ws1", "ws3", "ws2"):
        if getattr(a, k_ + "_lp") is not None:
            assert torch.equal(getattr(a, k_ + "_lp"), getattr(b, k_ + "_lp")), k_
    assert a.dw1.abs().max().item() > 0
