"""Expert-parallel training step over the C ABI's rank-local phases.

"AI Infra Kernel Lab", "Project status" (expert parallelism with a variable
All-to-All) and "Numerical contracts": the E experts are split over G ranks
(rank r owns experts [r L, r L + L), L = E / G).  Every rank routes its own
tokens; the dispatch exchange sends unweighted expert-major rows to each
expert's owner; the outputs return to their source rank, where the routing
weights are applied in the combine; the backward runs through both exchanges
in reverse.  Token shards may be uneven or empty.

This module plans the exchanges (which rows go where: index arithmetic on the
per-expert counts) and moves rows through a transport:

* ``TorchDistTransport``: one rank per process, ``torch.distributed``
  point-to-point sends and receives (NCCL between GPUs, gloo on CPU tensors),
  an all-gather of the counts and sum all-reduces of the small statistics;
* ``LocalTransport``: one process drives every rank (copies between the
  ranks' buffers); used to run and check the whole step on one device.

Every step of the layer's arithmetic runs in the library's kernels; this
module only allocates buffers, sums the small per-rank statistics, and moves
rows.
"""

from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

from . import binding as B


# ------------------------------------------------------------------ plan --

@dataclasses.dataclass(frozen=True)
class Block:
    """Rows of local expert ``l`` of rank ``dst`` that come from rank ``src``:
    rows [src_row, src_row + rows) of the source's expert-major buffer (all E
    experts) and [dst_row, dst_row + rows) of the owner's received rows."""
    src: int
    dst: int
    l: int
    src_row: int
    dst_row: int
    rows: int


class ExchangePlan:
    """The dispatch exchange of one step, from every rank's per-expert counts
    ``counts [G, E]`` (rank s routed counts[s, e] of its rows to expert e).

    A source's rows of expert e sit at [off_s[e], off_s[e] + counts[s, e]) of
    its expert-major buffer (off_s the exclusive scan of counts[s]).  The
    owner d of e keeps its local experts in order and, inside one expert,
    the rows of source 0, 1, ... one after the other: for the concatenation
    of the ranks' tokens this is exactly a single device's expert-major
    order."""

    def __init__(self, counts: np.ndarray):
        counts = np.asarray(counts, dtype=np.int64)
        G, E = counts.shape
        if E % G:
            raise ValueError("the ranks must divide the experts")
        self.G, self.E, self.L = G, E, E // G
        self.counts = counts
        self.src_offsets = np.zeros((G, E + 1), dtype=np.int64)
        self.src_offsets[:, 1:] = np.cumsum(counts, axis=1)
        # owner side: rows of local expert l, from every source
        per_expert = counts.sum(axis=0)                       # [E]
        self.recv_offsets = np.zeros((G, self.L + 1), dtype=np.int64)
        for d in range(G):
            self.recv_offsets[d, 1:] = np.cumsum(per_expert[d * self.L:(d + 1) * self.L])
        self.recv_rows = self.recv_offsets[:, -1].copy()      # [G]
        blocks = []
        for d in range(G):
            for l in range(self.L):
                e = d * self.L + l
                at = int(self.recv_offsets[d, l])
                for s in range(G):
                    n = int(counts[s, e])
                    if n:
                        blocks.append(Block(s, d, l, int(self.src_offsets[s, e]), at, n))
                    at += n
        # canonical order (source, owner, expert): every rank enumerates the
        # messages between a pair of ranks in the same order
        self.blocks = sorted(blocks, key=lambda b: (b.src, b.dst, b.l))

    def local_offsets(self, d: int) -> np.ndarray:
        return self.recv_offsets[d]


# ------------------------------------------------------------- transports --

class LocalTransport:
    """Every rank in this process: an exchange is a set of row copies between
    the ranks' buffers (on one device, in stream order), a sum all-reduce adds
    the ranks' tensors in rank order."""

    def __init__(self, world: int):
        self.world = world
        self.ranks = list(range(world))

    def all_gather_counts(self, counts: Dict[int, np.ndarray]) -> np.ndarray:
        return np.stack([np.asarray(counts[r], dtype=np.int64) for r in self.ranks])

    def all_reduce_sum(self, tensors: Dict[int, torch.Tensor]) -> None:
        total = tensors[self.ranks[0]].clone()
        for r in self.ranks[1:]:
            total += tensors[r]
        for r in self.ranks:
            tensors[r].copy_(total)

    def exchange(self, blocks: Sequence[Block], src_bufs: Dict[int, torch.Tensor],
                 dst_bufs: Dict[int, torch.Tensor], reverse: bool = False) -> None:
        for b in blocks:
            if not reverse:
                dst_bufs[b.dst][b.dst_row:b.dst_row + b.rows].copy_(
                    src_bufs[b.src][b.src_row:b.src_row + b.rows])
            else:
                dst_bufs[b.src][b.src_row:b.src_row + b.rows].copy_(
                    src_bufs[b.dst][b.dst_row:b.dst_row + b.rows])


class TorchDistTransport:
    """This process is one rank of an initialised ``torch.distributed`` group;
    rows move by point-to-point sends and receives batched per exchange
    (NCCL on GPU tensors, gloo on CPU tensors)."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.ranks = [self.rank]

    def all_gather_counts(self, counts: Dict[int, np.ndarray]) -> np.ndarray:
        mine = torch.as_tensor(np.asarray(counts[self.rank], dtype=np.int64))
        dev = self._device()
        mine = mine.to(dev)
        out = [torch.empty_like(mine) for _ in range(self.world)]
        self.dist.all_gather(out, mine, group=self.group)
        return torch.stack(out).cpu().numpy()

    def all_reduce_sum(self, tensors: Dict[int, torch.Tensor]) -> None:
        self.dist.all_reduce(tensors[self.rank], group=self.group)

    def exchange(self, blocks: Sequence[Block], src_bufs: Dict[int, torch.Tensor],
                 dst_bufs: Dict[int, torch.Tensor], reverse: bool = False) -> None:
        me = self.rank
        ops = []
        for b in blocks:
            s, d = (b.src, b.dst) if not reverse else (b.dst, b.src)
            s_row, d_row = (b.src_row, b.dst_row) if not reverse else (b.dst_row, b.src_row)
            if s == me and d == me:
                dst_bufs[d][d_row:d_row + b.rows].copy_(src_bufs[s][s_row:s_row + b.rows])
            elif s == me:
                ops.append(self.dist.P2POp(self.dist.isend, src_bufs[s][s_row:s_row + b.rows],
                                           d, self.group))
            elif d == me:
                ops.append(self.dist.P2POp(self.dist.irecv, dst_bufs[d][d_row:d_row + b.rows],
                                           s, self.group))
        if ops:
            for w in self.dist.batch_isend_irecv(ops):
                w.wait()

    def _device(self):
        backend = self.dist.get_backend(self.group)
        return torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else "cpu"


# ------------------------------------------------------------------ ranks --

class EPRank:
    """One rank's share of an expert-parallel MoE layer: the replicated router
    (fp32 master), the fp32 masters (and bf16 copies) of its L local experts,
    its workspace, and this step's received rows."""

    def __init__(self, rank: int, n_ranks: int, T: int, T_total: int, D, F, E, k, act, score,
                 dtype, has_bias, aux_alpha, w_gate, w1, w2, w3=None, b1=None, b2=None,
                 logit_bias=None, corr_bias=None, n_groups=1, topk_groups=1,
                 group_score="top2_sum", device="cuda", store_grads=True):
        if E % n_ranks:
            raise ValueError("the ranks must divide the experts")
        self.rank, self.n_ranks, self.dtype = rank, n_ranks, dtype
        self.L = E // n_ranks
        self.device = torch.device(device)
        self.cfg = B.make_config(T, D, F, E, k, act=act, score=score, n_groups=n_groups,
                                 topk_groups=topk_groups, group_score=group_score, dtype=dtype,
                                 has_bias=has_bias, aux_alpha=aux_alpha)
        self.ep = B.moe_ep_config(n_ranks, rank, T_total)
        dev = self.device
        lo, hi = rank * self.L, (rank + 1) * self.L

        def f32(t, local=False):
            if t is None:
                return None
            t = t[lo:hi] if local else t
            return t.detach().to(dev, torch.float32).contiguous().clone()

        self.w_gate, self.logit_bias, self.corr_bias = f32(w_gate), f32(logit_bias), f32(corr_bias)
        self.w1, self.w2, self.w3 = f32(w1, True), f32(w2, True), f32(w3, True)
        self.b1, self.b2 = f32(b1, True), f32(b2, True)
        lp = dtype == "bf16"
        cast = lambda t: None if t is None or not lp else t.to(torch.bfloat16).contiguous()  # noqa: E731
        self.w1_lp, self.w2_lp, self.w3_lp = cast(self.w1), cast(self.w2), cast(self.w3)
        keep = store_grads or not lp
        z = lambda t, need=False: None if t is None or not (keep or need) else torch.zeros_like(t)  # noqa: E731
        self.dw1, self.dw2, self.dw3 = z(self.w1), z(self.w2), z(self.w3)
        self.db1, self.db2 = z(self.b1, True), z(self.b2, True)   # biases always need buffers
        self.workspace = torch.empty(max(B.moe_ep_workspace_size(self.cfg, self.ep), 1),
                                     dtype=torch.uint8, device=dev)
        if B.moe_ep_workspace_size(self.cfg, self.ep) == 0:
            raise B.MoEError("moe_ep_workspace_size", B.MOE_ERR_INVALID_ARG, "invalid request")
        self.offs = B.moe_ep_buffer_offsets(self.cfg, self.ep)
        self.score_sum = torch.zeros(E, dtype=torch.float32, device=dev)
        self.counts_total = torch.zeros(E, dtype=torch.int32, device=dev)
        self.d_loss = torch.zeros(2, dtype=torch.float32, device=dev)
        self.dw_gate = torch.zeros(E, D, dtype=torch.float32, device=dev)
        self.status = torch.zeros(4, dtype=torch.int32, device=dev)
        self.rows = 0
        self.x = self.target = None

    # expert-major views of the workspace (all E experts, this rank's tokens)
    def _ws_rows(self, which: int) -> torch.Tensor:
        c = self.cfg
        dt = torch.bfloat16 if self.dtype == "bf16" else torch.float32
        es = 2 if self.dtype == "bf16" else 4
        n = c.T * c.k * c.D * es
        start = self.offs[which]
        return self.workspace[start:start + max(n, es)].view(dt)[: c.T * c.k * c.D].view(
            c.T * c.k, c.D)

    @property
    def xe(self):
        return self._ws_rows(0)

    @property
    def ye(self):
        return self._ws_rows(1)

    @property
    def dye(self):
        return self._ws_rows(2)

    @property
    def dxe(self):
        return self._ws_rows(3)

    def router_weights(self):
        return B.make_weights(self.w_gate, None, None, logit_bias=self.logit_bias,
                              corr_bias=self.corr_bias)

    def expert_weights(self):
        lp = self.dtype == "bf16"
        return B.make_weights(None, self.w1_lp if lp else self.w1, self.w2_lp if lp else self.w2,
                              self.w3_lp if lp else self.w3, self.b1, self.b2)

    def expert_params(self):
        g = B.make_grads(None, self.dw1, self.dw2, self.dw3, self.db1, self.db2)
        return B.make_params(None, self.w1, self.w2, g, w3=self.w3, b1=self.b1, b2=self.b2,
                             w1_lp=self.w1_lp, w3_lp=self.w3_lp, w2_lp=self.w2_lp)

    def counts(self) -> np.ndarray:
        c = self.cfg
        out = torch.empty(c.E, dtype=torch.int32, device=self.device)
        B.moe_ep_get_routing(c, self.ep, self.workspace, counts=out)
        return out.cpu().numpy().astype(np.int64)

    def routing(self) -> dict:
        """This rank's routing of its tokens over all E experts."""
        c = self.cfg
        dev = self.device
        R = c.T * c.k
        out = dict(scores=torch.empty(max(c.T, 1), c.E, device=dev),
                   idx=torch.empty(max(c.T, 1), c.k, dtype=torch.int32, device=dev),
                   counts=torch.empty(c.E, dtype=torch.int32, device=dev),
                   offsets=torch.empty(c.E + 1, dtype=torch.int32, device=dev),
                   slot_of=torch.empty(max(c.T, 1), c.k, dtype=torch.int32, device=dev))
        B.moe_ep_get_routing(c, self.ep, self.workspace, **out)
        out["scores"], out["idx"], out["slot_of"] = (out["scores"][:c.T], out["idx"][:c.T],
                                                     out["slot_of"][:c.T])
        return out

    def alloc_rows(self, rows: int, offsets: np.ndarray):
        c = self.cfg
        dev = self.device
        dt = torch.bfloat16 if self.dtype == "bf16" else torch.float32
        n = max(rows, 1)
        swiglu = c.act == B.ACT["swiglu"]
        self.rows = rows
        self.r_offsets = torch.as_tensor(np.asarray(offsets, dtype=np.int32)).to(dev)
        self.r_x = torch.empty(n, c.D, dtype=dt, device=dev)
        self.r_h1 = torch.empty(n, c.F, dtype=dt, device=dev)
        self.r_h3 = torch.empty(n, c.F, dtype=dt, device=dev) if swiglu else None
        self.r_a = torch.empty(n, c.F, dtype=dt, device=dev)
        self.r_y = torch.empty(n, c.D, dtype=dt, device=dev)
        self.r_dy = torch.empty(n, c.D, dtype=dt, device=dev)
        self.r_dh1 = torch.empty(n, c.F, dtype=dt, device=dev)
        self.r_dh3 = torch.empty(n, c.F, dtype=dt, device=dev) if swiglu else None
        self.r_dx = torch.empty(n, c.D, dtype=dt, device=dev)
        # fp32 layers: scratch that puts the expert GEMMs on the tensor cores,
        # as the single-device step's workspace does
        nbytes = B.moe_ep_f32_scratch_size(c, self.ep, rows)
        self.r_f32 = torch.empty(nbytes, dtype=torch.uint8, device=dev) if nbytes else None

    def ep_rows(self):
        return B.make_ep_rows(self.rows, self.r_offsets, self.r_x, self.r_h1, self.r_h3, self.r_a,
                              self.r_y, self.r_dy, self.r_dh1, self.r_dh3, self.r_dx, self.status,
                              self.r_f32)


def train_step(ranks: List[EPRank], transport, xs: Dict[int, torch.Tensor],
               targets: Dict[int, torch.Tensor], lr: float,
               dxs: Optional[Dict[int, torch.Tensor]] = None) -> Dict[str, float]:
    """One expert-parallel training step for the ranks this process drives
    (all of them with ``LocalTransport``, its own with ``TorchDistTransport``).
    ``xs[r]`` [T_r, D] in the layer dtype, ``targets[r]`` [T_r, D] fp32;
    ``dxs[r]`` receives dL/dx of rank r's tokens when given.  Returns the
    losses (the same on every rank)."""
    me = {rk.rank: rk for rk in ranks}
    # 1. route every rank's own tokens; share the counts; sum the score sums
    for rk in ranks:
        rk.x, rk.target = xs[rk.rank], targets[rk.rank]
        B.moe_ep_route(rk.cfg, rk.ep, rk.router_weights(), rk.x, rk.score_sum, rk.workspace)
    counts = transport.all_gather_counts({r: rk.counts() for r, rk in me.items()})
    plan = ExchangePlan(counts)
    transport.all_reduce_sum({r: rk.score_sum for r, rk in me.items()})
    totals = torch.as_tensor(counts.sum(axis=0).astype(np.int32))
    for rk in ranks:
        rk.counts_total.copy_(totals)
        rk.alloc_rows(int(plan.recv_rows[rk.rank]), plan.local_offsets(rk.rank))
        rk.status.zero_()
    # 2. dispatch: unweighted rows to the experts' owners
    transport.exchange(plan.blocks, {r: rk.xe for r, rk in me.items()},
                       {r: rk.r_x for r, rk in me.items()})
    # 3. local experts forward
    for rk in ranks:
        B.moe_ep_expert_forward(rk.cfg, rk.ep, rk.expert_weights(), rk.ep_rows())
    # 4. outputs back to their sources
    transport.exchange(plan.blocks, {r: rk.r_y for r, rk in me.items()},
                       {r: rk.ye for r, rk in me.items()}, reverse=True)
    # 5. combine (gates applied at the source), losses, combine backward
    for rk in ranks:
        B.moe_ep_combine(rk.cfg, rk.ep, rk.counts_total, rk.score_sum, rk.target, rk.d_loss,
                         rk.workspace)
    # 6. output gradients to the owners
    transport.exchange(plan.blocks, {r: rk.dye for r, rk in me.items()},
                       {r: rk.r_dy for r, rk in me.items()})
    # 7. local experts backward + SGD
    for rk in ranks:
        B.moe_ep_expert_backward(rk.cfg, rk.ep, rk.expert_params(), rk.ep_rows(), lr)
    # 8. input gradients back to their sources
    transport.exchange(plan.blocks, {r: rk.r_dx for r, rk in me.items()},
                       {r: rk.dxe for r, rk in me.items()}, reverse=True)
    # 9. router backward of each rank's tokens; 10. sum dW_g, update the router
    for rk in ranks:
        dx = None if dxs is None else dxs.get(rk.rank)
        B.moe_ep_router_backward(rk.cfg, rk.ep, rk.w_gate, rk.x, rk.dw_gate, dx, rk.workspace)
    transport.all_reduce_sum({r: rk.dw_gate for r, rk in me.items()})
    for rk in ranks:
        B.moe_ep_router_update(rk.cfg, rk.w_gate, rk.dw_gate, lr)
    # losses: the MSE shares summed over the ranks; aux is the same everywhere
    mse = {r: rk.d_loss[:1].clone() for r, rk in me.items()}
    transport.all_reduce_sum(mse)
    first = ranks[0]
    return {"mse": float(mse[first.rank].item()), "aux": float(first.d_loss[1].item()),
            "rows_received": {rk.rank: rk.rows for rk in ranks}}
