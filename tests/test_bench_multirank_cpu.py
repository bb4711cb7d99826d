"""The multi-rank host logic of bench.py on CPU (gloo, world size 2): the
cross-rank barrier and max, the whole-job rate, and the reference arm under
torchrun (rank 0 alone prints one JSON line, the other ranks exit 0)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, ws, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(ws), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench

    world, r, local = bench.dist_setup()
    assert (world, r, local) == (ws, rank, rank)
    bench.barrier(world)
    # each rank "measured" a different time; the job time is the slowest
    ms = 10.0 + 5.0 * rank
    ms_max = bench.max_over_ranks(ms, world)
    out[rank] = (ms_max, bench.job_rate(steps=100, ms_max=ms_max, world=world))
    import torch.distributed as dist

    dist.destroy_process_group()


def test_barrier_max_and_job_rate_with_two_gloo_ranks():
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == out[1]
    ms_max, rate = out[0]
    assert ms_max == 15.0
    assert rate == pytest.approx(2 * 100 / 15e-3)  # tokens of both ranks / slowest time


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--steps", "1", "--warmup", "1", "--reference-budget", "5"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["e2e"]["h2d_bytes_per_step"] == 0
