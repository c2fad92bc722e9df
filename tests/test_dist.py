"""The N > 1 path on the CPU: bench.py runs one replica of the step per GPU
(the path has no exchange: every head is independent), takes the slowest
rank's time and reports the work of all ranks over it.  These tests run
world-size-2 gloo groups on the CPU; nothing here touches a GPU."""

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
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, local_ms, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    ms = bench.max_over_ranks(local_ms[rank], ws, "cpu")
    out[rank] = (ms, bench.job_throughput(1e12, ws, ms))
    dist.barrier()
    dist.destroy_process_group()


def test_slowest_rank_sets_the_job_time():
    """Every rank gets the slowest rank's step time; the job's throughput is
    the work of both ranks over that time (weak scaling)."""
    ws, port = 2, _free_port()
    local_ms = [0.25, 0.40]
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(ws, port, local_ms, out), nprocs=ws, join=True, start_method="spawn")
        res = dict(out)
    for rank in range(ws):
        ms, tf = res[rank]
        assert ms == pytest.approx(0.40)
        assert tf == pytest.approx(2 * 1e12 / 0.40e-3 / 1e12)


def test_single_rank_is_unchanged():
    import bench
    assert bench.max_over_ranks(0.3, 1, "cpu") == 0.3
    assert bench.job_throughput(1e12, 1, 1.0) == pytest.approx(1000.0)


def test_reference_arm_prints_once_under_torchrun():
    """bench.py --impl reference under a 2-rank launch: rank 0 alone times the
    oracle and prints one JSON line; the other rank exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
