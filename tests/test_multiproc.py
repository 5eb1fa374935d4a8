"""The multi-process side of bench.py on the host (gloo, world size 2): the job's time is the
slowest rank's, the job's value counts every rank's tokens, and under torchrun the reference arm
prints one line from rank 0 while the other rank exits cleanly. The attention itself has no
exchange step (tokens are independent): several GPUs run replicas."""
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


def _rank(rank, world, port, values, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench

    q.put((rank, bench.max_over_ranks(values[rank], world)))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    values = [12.5, 31.25]
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, values, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert got == {0: 31.25, 1: 31.25}


def test_job_value_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.job_value(1, 256, 10, 1.0) == pytest.approx(2_560_000.0)
    assert bench.job_value(2, 256, 10, 2.0) == pytest.approx(2_560_000.0)  # twice the tokens, twice the time
    assert bench.max_over_ranks(7.0, 1) == 7.0


def test_reference_arm_under_torchrun_world2():
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2", "--master-addr",
           "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference", "--config", "1",
           "--steps", "1", "--warmup", "3", "--gpus", "2"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0
