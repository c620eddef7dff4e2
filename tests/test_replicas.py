"""The multi-GPU path is replicas only (every rank runs the whole workload, no data-path
collective): its timing aggregation and launch, tested with world_size 2 on CPU (gloo)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks_of(dist, times[rank])
        out.put((rank, ms, bench.whole_job_rate(world, bench.COUNT, ms)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    times = [1.25, 2.5]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, ms, rate in res:
        assert ms == 2.5  # the slowest rank sets the time
        assert rate == pytest.approx(2 * 24 / 2.5e-3)


def test_no_process_group_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks_of(None, 3.0) == 3.0
    assert bench.whole_job_rate(1, 24, 2.0) == pytest.approx(12000.0)


def test_reference_arm_under_torchrun_world2():
    """torchrun with two ranks: rank 0 alone times the oracle and prints one JSON line."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    # the same workload description as the GPU arm's line
    sys.path.insert(0, ROOT)
    import bench
    assert d["config"] == bench.bench_config(2)
