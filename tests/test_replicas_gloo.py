"""The N > 1 path of bench.py on CPU: world-size-2 gloo ranks.

Every rank runs its own replica of the step (the layer has no exchange
step), so the only cross-rank work is the timing reduction: the slowest
rank's time, and whole-job throughput = all ranks' tokens over that time.
The reference arm runs on rank 0 only; other ranks exit 0 without output."""

import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(times[rank], "cpu")
        rate = bench.whole_job_rate(1000, world, 5, slowest)
        q.put((rank, slowest, rate))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_gloo():
    world, times = 2, [0.25, 0.4]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, slowest, rate in got:
        assert slowest == max(times)
        assert abs(rate - 1000 * world * 5 / max(times)) < 1e-9


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.125, "cpu") == 0.125
    assert bench.whole_job_rate(64, 1, 4, 2.0) == 128.0


def _reference_arm(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
               MASTER_ADDR="127.0.0.1")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--workload", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "0"],
                          env=env, capture_output=True, text=True, timeout=300)


def test_reference_arm_rank0_only():
    r1 = _reference_arm(1)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = _reference_arm(0)
    assert r0.returncode == 0, r0.stderr
    lines = [ln for ln in r0.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
