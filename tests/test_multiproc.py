"""The multi-rank host path of bench.py on CPU (gloo, world size 2).

The block needs no exchange at EP=1, so N GPUs run N independent replicas;
what the ranks share is the timing protocol: a barrier around the timed
region, the slowest rank's time, and the whole-job throughput.  These tests
run that logic with two gloo ranks on the CPU, and the reference arm under
torchrun (rank 0 prints one line, the other rank exits quietly).
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        my_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
        ms = bench.reduce_max(my_ms, world)
        out[rank] = (ms, bench.aggregate(rows_per_rank=1000, ms_max=ms, ws=world))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_time_and_whole_job_rate():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1]
    ms, rate = out[0]
    assert ms == 15.0                          # the slowest rank
    assert rate == pytest.approx(2 * 1000 / 0.015)   # all rows over that time


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--config", "c0", "--steps", "2", "--warmup", "1", "--gpus", "2"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["value"] > 0 and line["unit"] == "rows/s"
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
