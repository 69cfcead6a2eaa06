"""The expert-parallel exchanges on CPU: the planning of ``expert_parallel``
and its ``torch.distributed`` transport on world-size-2 gloo ranks.

"AI Infra Kernel Lab", "Project status" (expert parallelism over a variable
All-to-All, verified there on Gloo) and "Numerical contracts" (unweighted rows
dispatched to the experts' owners, outputs returned to their source rank,
uneven and empty token shards).  Each row carries a tag (its global token id
and top-k position), so a test checks exactly where every row lands:

* after the dispatch exchange an owner holds, for each local expert, the rows
  the oracle's dispatch of the CONCATENATED tokens gives that expert, in the
  same order (source rank order = global token order);
* after the return exchange every source row holds the value its owner wrote
  for it;
* shards may be empty and experts may receive nothing.
"""

import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from oracle import moe_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _routing(shards, E, k, seed):
    """Per-rank top-k expert ids (distinct per token), skewed, with the last
    expert never chosen."""
    rng = np.random.default_rng(seed)
    p = rng.dirichlet(np.full(E, 0.7))
    p[-1] = 0.0
    p /= p.sum()
    return [np.array([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)],
                     dtype=np.int32).reshape(T, k) for T in shards]


def _source_rows(idx_r, base, E, D):
    """A source's expert-major rows (all E experts), each tagged with its
    global token id and top-k position: column 0 = token, 1 = j, the rest a
    function of both."""
    counts, offsets, src_tok, src_j, _ = O.dispatch(idx_r, E)
    R = int(offsets[-1])
    rows = np.zeros((R, D))
    rows[:, 0] = base + src_tok
    rows[:, 1] = src_j
    for c in range(2, D):
        rows[:, c] = (base + src_tok) * 7 + src_j * 3 + c
    return counts, torch.from_numpy(rows)


def _expected_owner_rows(idx_all, E, G, d, D):
    """The rows of owner d's experts under a single device's dispatch of all
    tokens, in that order."""
    L = E // G
    _, offsets, src_tok, src_j, _ = O.dispatch(idx_all, E)
    lo, hi = int(offsets[d * L]), int(offsets[(d + 1) * L])
    return src_tok[lo:hi], src_j[lo:hi]


def _check_rank(rank, transport, shards, E, k, D, seed):
    from sparse_mixture_experts_softmax_gb300.expert_parallel import ExchangePlan
    G = len(shards)
    idx = _routing(shards, E, k, seed)
    base = int(sum(shards[:rank]))
    counts, src = _source_rows(idx[rank], base, E, D)
    plan = ExchangePlan(transport.all_gather_counts({rank: counts}))
    recv = torch.full((max(int(plan.recv_rows[rank]), 1), D), -1.0, dtype=torch.float64)
    transport.exchange(plan.blocks, {rank: src}, {rank: recv})
    tok, j = _expected_owner_rows(np.concatenate(idx), E, G, rank, D)
    n = int(plan.recv_rows[rank])
    assert n == len(tok)
    np.testing.assert_array_equal(recv[:n, 0].numpy(), tok)
    np.testing.assert_array_equal(recv[:n, 1].numpy(), j)
    # per-expert segments the owner's GEMMs use
    L = E // G
    tot = np.concatenate(idx)
    for l in range(L):
        e = rank * L + l
        assert plan.recv_offsets[rank, l + 1] - plan.recv_offsets[rank, l] == (tot == e).sum()
    # return: the owner writes f(row) back; every source row gets f of itself
    back = recv * 2.0 + 1.0
    got = torch.full_like(src, -1.0)
    transport.exchange(plan.blocks, {rank: back}, {rank: got}, reverse=True)
    np.testing.assert_array_equal(got.numpy(), src.numpy() * 2.0 + 1.0)
    return n


def _gloo_main(rank, world, port, shards, E, k, D, seed, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from sparse_mixture_experts_softmax_gb300.expert_parallel import TorchDistTransport
        n = _check_rank(rank, TorchDistTransport(), shards, E, k, D, seed)
        q.put((rank, n, None))
    except Exception as e:   # reported to the parent
        q.put((rank, -1, repr(e)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("shards,E,k", [((57, 23), 8, 2), ((0, 41), 6, 3), ((64, 0), 8, 3)])
def test_exchanges_on_two_gloo_ranks(shards, E, k):
    world, D = 2, 5
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gloo_main, args=(r, world, port, shards, E, k, D, 11, q))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, n, err in got:
        assert err is None, (rank, err)
    # every routed row went to exactly one owner
    assert sum(n for _, n, _ in got) == sum(shards) * k


@pytest.mark.parametrize("shards,E", [((30, 0, 17), 6), ((5, 9, 0, 12), 8)])
def test_local_transport_matches_the_oracle_dispatch(shards, E):
    """The same checks with one process driving every rank (the transport
    the single-device run of the whole step uses)."""
    from sparse_mixture_experts_softmax_gb300.expert_parallel import ExchangePlan, LocalTransport
    G, k, D = len(shards), 2, 4
    idx = _routing(shards, E, k, 5)
    tr = LocalTransport(G)
    srcs, counts = {}, {}
    for r in range(G):
        counts[r], srcs[r] = _source_rows(idx[r], int(sum(shards[:r])), E, D)
    plan = ExchangePlan(tr.all_gather_counts(counts))
    recvs = {r: torch.full((max(int(plan.recv_rows[r]), 1), D), -1.0, dtype=torch.float64)
             for r in range(G)}
    tr.exchange(plan.blocks, srcs, recvs)
    for d in range(G):
        tok, j = _expected_owner_rows(np.concatenate(idx), E, G, d, D)
        n = int(plan.recv_rows[d])
        np.testing.assert_array_equal(recvs[d][:n, 0].numpy(), tok)
        np.testing.assert_array_equal(recvs[d][:n, 1].numpy(), j)
    outs = {r: torch.full_like(srcs[r], -1.0) for r in range(G)}
    tr.exchange(plan.blocks, {d: recvs[d] * 3.0 for d in range(G)}, outs, reverse=True)
    for r in range(G):
        np.testing.assert_array_equal(outs[r].numpy(), srcs[r].numpy() * 3.0)
    # sums over ranks in rank order
    ts = {r: torch.tensor([float(r + 1), 2.0 * r]) for r in range(G)}
    tr.all_reduce_sum(ts)
    for r in range(G):
        assert ts[r].tolist() == [G * (G + 1) / 2, float(G * (G - 1))]


def test_plan_rejects_ranks_that_do_not_divide_the_experts():
    from sparse_mixture_experts_softmax_gb300.expert_parallel import ExchangePlan
    with pytest.raises(ValueError):
        ExchangePlan(np.zeros((3, 8), dtype=np.int64))
