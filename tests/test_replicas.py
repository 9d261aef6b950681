"""Multi-GPU is replicas only: every rank drafts and verifies its own requests and the
job rate is all ranks' steps over the slowest rank's time.  The host logic runs here on
CPU with the gloo backend at world size 2."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
    m = bench.max_over_ranks(local_ms, world)
    rate = bench.whole_job_rate(100, world, m / 1000.0)
    seeds = [bench.replica_step_seed(s, rank) for s in range(4)]
    out.put((rank, m, rate, seeds))
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_take_the_max_over_ranks_and_distinct_inputs():
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
    for rank, m, rate, _ in res:
        assert m == 15.0
        assert abs(rate - 2 * 100 / 0.015) < 1e-6
    assert not set(res[0][3]) & set(res[1][3])


def test_reference_arm_under_torchrun_prints_one_line():
    """torchrun with 2 ranks: rank 0 times the oracle and prints one JSON line, rank 1
    exits without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--config", "tiny", "--gpus", "2", "--steps", "2", "--warmup", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
