"""The multi-rank path of bench.py on CPU: world-size-2 gloo ranks (the GPU
pool has one GPU per box, so N > 1 is only ever replicas; its host logic --
rendezvous, barrier, max over ranks, whole-job aggregation, rank-0-only
reference arm -- is checked here)."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench as b
    import torch.distributed as dist
    w, r, _ = b.dist_init()
    b.dist_barrier(w)
    slowest = b.dist_max(10.0 + 5.0 * r, w)
    # the reference arm: rank 0 alone does work
    class A:
        warmup, steps = 0, 0
    line, _ = b.run_reference(A, w, r) if r != 0 else (None, r)
    b.dist_barrier(w)
    dist.destroy_process_group()
    q.put((r, w, dist.is_available(), slowest, line))


def test_two_gloo_ranks_barrier_and_max():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, *_ in res] == [0, 1]
    assert all(w == 2 for _, w, *_ in res)
    assert all(s == 15.0 for *_, s, _ in res)          # max over ranks reaches every rank
    assert res[1][4] is None                            # rank 1 does no reference work


def test_whole_job_throughput_is_weak_scaling_aggregate():
    one = bench.throughput_gbs(1e9, 10, 1, 1000.0)
    assert one == pytest.approx(10.0)
    assert bench.throughput_gbs(1e9, 10, 4, 1000.0) == pytest.approx(4 * one)
    assert bench.throughput_gbs(1e9, 10, 4, 2000.0) == pytest.approx(2 * one)   # slowest rank decides


def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
