"""The benchmark's multi-rank host logic on CPU: two gloo ranks.

The path has no exchange step, so N GPUs run N replicas; what needs covering
is the launch, the barrier, the max-over-ranks timing and the whole-job
aggregate, and that only rank 0 prints. The GPU arm cannot run here; the
reference arm (the oracle on the host cores) can, under torchrun.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist = bench.dist_init(world)
    try:
        # rank r "measured" 10 + r ms; every rank must see the slowest one
        ms = bench.max_over_ranks(dist, 10.0 + rank)
        v = bench.aggregate_gbs(world, 1e9, ms)
        dist.barrier()
        out.put((rank, ms, v))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [11.0, 11.0]
    # 2 ranks x 1 GB each over 11 ms
    assert all(abs(r[2] - 2 * 1e9 / 11e-3 / 1e9) < 1e-6 for r in res)


def test_single_rank_helpers_are_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_init(1) is None
    assert bench.max_over_ranks(None, 3.5) == 3.5
    assert bench.aggregate_gbs(1, 2e9, 1000.0) == pytest.approx(2.0)


def test_reference_arm_two_ranks_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
