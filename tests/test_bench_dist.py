"""The bench's multi-rank path on CPU with gloo (world size 2).

The decode path shards by sequence with no exchange, so N GPUs run N replicas;
what the ranks share is the timing: a barrier on both sides and the slowest
rank's time.  These tests run that logic on CPU processes."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(1.0 + rank * 0.5, dist, torch.device("cpu"))
        dist.barrier()
        q.put((rank, slowest, bench.job_throughput(world, 4e9, slowest)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_throughput():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, gbs in res:
        assert slowest == 1.5                              # every rank sees the slowest rank's time
        assert gbs == pytest.approx(2 * 4e9 / 1.5e-3 / 1e9)  # both ranks' bytes over that time


def test_single_rank_helpers_need_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, None, None) == 3.25
    assert bench.job_throughput(1, 1e9, 1.0) == pytest.approx(1000.0)


def test_reference_arm_under_torchrun_two_ranks():
    """Rank 0 alone prints the reference line; the other rank exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "1", "--gpus", "2", "--steps", "3", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_main_reads_no_deleted_name():
    """Names that main() deletes (the extras free the headline runner's cache) are not read
    afterwards on the same path: the default run, extras included, reaches its JSON line."""
    import ast
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    main = next(n for n in tree.body if isinstance(n, ast.FunctionDef) and n.name == "main")
    deleted = {}
    for node in ast.walk(main):
        if isinstance(node, ast.Delete):
            for t in node.targets:
                if isinstance(t, ast.Name):
                    deleted[t.id] = max(deleted.get(t.id, 0), node.lineno)
    late = [(n.id, n.lineno) for n in ast.walk(main)
            if isinstance(n, ast.Name) and isinstance(n.ctx, ast.Load) and n.id in deleted
            and n.lineno > deleted[n.id]]
    assert not late, late
