"""The benchmark's multi-process path on the CPU: two gloo ranks (one replica
per GPU in a real run) share only a barrier and the max of their timings;
the reference arm prints from rank 0 alone."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from tests.conftest import ROOT


def _worker(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    ctx = bench.DistCtx()
    ctx.barrier()
    got = ctx.max(float(10 * (rank + 1)))  # each rank "timed" a different duration
    ctx.barrier()
    out_q.put((rank, ctx.world, got))
    ctx.close()


def _free_port():
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_two_ranks_share_barrier_and_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for pr in procs:
        pr.start()
    for pr in procs:
        pr.join(timeout=120)
        assert pr.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    # both ranks see world 2 and the max over ranks (20.0)
    assert res == [(0, 2, 20.0), (1, 2, 20.0)]


def test_reference_arm_under_two_ranks_prints_once():
    """bench.py --impl reference under torchrun: rank 0 prints one JSON line,
    the other rank exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--workload", "p4_n4099_f32"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["value"] > 0
