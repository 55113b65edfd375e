"""The benchmark's multi-process host logic on CPU, world size 2 over gloo:
replicas report the max over ranks of the timed region and the sum of the
tokens all ranks decoded; under torchrun the reference arm runs on rank 0
alone (one JSON line, the other rank exits 0)."""
import json
import os
import socket
import subprocess
import sys
from pathlib import Path

import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parents[1]


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, str(ROOT))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, _ = bench.dist_env()
        ms = [12.5, 17.0][rank]          # per-rank timed region
        tokens = [256.0, 256.0][rank]    # tokens each replica decoded
        q.put((r, w, bench.aggregate_max(ms, w), bench.aggregate_sum(tokens, w)))
    finally:
        dist.destroy_process_group()


def test_replica_aggregation_gloo():
    world, port = 2, free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, (r, w, mx, tot) in enumerate(got):
        assert (r, w) == (rank, world)
        assert mx == 17.0 and tot == 512.0
    # whole-job value: tokens of all ranks over the slowest rank's time
    assert got[0][3] / (got[0][2] / 1e3) == 512.0 / 0.017


def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), str(ROOT / "bench.py"),
           "--impl", "reference", "--workload", "tiny", "--gpus", "2", "--steps", "2", "--warmup", "3"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0
