"""The N > 1 launch path of bench.py, on CPU with the gloo backend (world size 2).

The layer has no exchange between GPUs: all P ranks of the method are virtual
shards on one GPU, so `bench.py --gpus N` runs N independent replicas. What
the launch path adds on top is host logic: the job's time is the slowest
rank's (a max over ranks), the job's throughput counts every rank's tokens,
and only rank 0 prints. These tests run that logic in two processes.
"""
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


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + 5.0 * rank                  # the ranks' own timed regions, ms
        job = bench.max_over_ranks(mine, "cpu", world)
        out[rank] = (job, bench.job_tokens_per_s(4096, 3, world, job))
    finally:
        dist.destroy_process_group()


def test_job_time_is_the_slowest_rank_and_throughput_counts_all_ranks():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]                         # every rank sees the job's figures
    job, value = res[0]
    assert job == 15.0
    assert value == pytest.approx(4096 * 3 * world / 0.015)


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5, "cpu", 1) == 7.5
    assert bench.job_tokens_per_s(100, 2, 1, 10.0) == pytest.approx(20000.0)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    """`--impl reference` with two ranks: rank 0 times the oracle and prints; rank 1 exits 0."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "3", "--workload", "tiny", "--ref-sl", "64"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    p = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["config"]["workload"] == "tiny"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["value"] > 0
