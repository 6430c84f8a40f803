"""The multi-rank path of bench.py on CPU: two gloo ranks, each timing its own
replica; the job time is the maximum over ranks and the whole-job rate counts
every rank's units (weak scaling).  No GPU and no collective on the data path."""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local = [12.5, 30.0][rank]                      # rank 1 is the slow one
    job = bench.job_time_ms(local, world, torch.device("cpu"))
    rate = bench.whole_job_rate(3926, world, 4, job)
    out[rank] = (job, rate)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_job_time_is_max_and_rate_counts_all_ranks():
    mgr = mp.Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_rank, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert out[0][0] == out[1][0] == 30.0
    assert out[0][1] == out[1][1] == pytest.approx(2 * 4 * 3926 / 0.030)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_time_ms(7.0, 1, torch.device("cpu")) == 7.0
    assert bench.whole_job_rate(100, 1, 10, 1000.0) == pytest.approx(1000.0)


def test_reference_arm_prints_one_line_on_rank0_only():
    import json
    import subprocess
    env = dict(os.environ)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], capture_output=True, text=True,
                       timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tok/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0
    env.update(RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], capture_output=True, text=True,
                       timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0 and r.stdout.strip() == ""
