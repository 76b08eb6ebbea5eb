"""The N > 1 path on the CPU (gloo, world size 2): ranks are independent replicas, so the only
cross-rank step is the max-over-ranks timing that bench.py reduces, and the reference arm runs on
rank 0 alone."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sys.path.insert(0, ROOT)
        import bench
        local = [3.0, 5.0][rank]                       # per-rank timed milliseconds
        ms = bench.max_over_ranks(local, world, "cpu")
        q.put((rank, ms, bench.job_tokens_per_s(world, 4096, 10, ms)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, tps in got:
        assert ms == 5.0                               # every rank sees the slowest one
        assert tps == pytest.approx(2 * 4096 * 10 / 5e-3)


def test_single_rank_aggregation_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, 1, "cpu") == 2.5
    assert bench.job_tokens_per_s(1, 256, 4, 2.0) == pytest.approx(256 * 4 / 2e-3)


def test_reference_arm_prints_once_under_torchrun():
    """`bench.py --impl reference` under a two-rank launch: rank 0 prints one JSON line, rank 1
    exits 0 without work (the oracle runs on the host cores; no GPU is needed)."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--config", "tiny_f32", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    res = json.loads(lines[0])
    assert res["impl"] == "reference" and res["n_gpus"] == 2 and res["value"] > 0
