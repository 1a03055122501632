"""The N > 1 path of bench.py on the host: world-size-2 gloo ranks on the CPU.

Each rank runs its own copy of the workload (the (batch, head) problems are
independent, so the path shards with no data-path collective); only the timing
is reduced: the slowest rank's time, and the whole-job throughput is the work
of all ranks divided by it.  The reference arm under torchrun runs on rank 0
alone and prints exactly one line.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(10.0 + 5.0 * rank)
        out.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    mp.start_processes(_rank_main, args=(2, free_port(), q), nprocs=2, join=True, start_method="spawn")
    res = dict(q.get() for _ in range(2))
    assert res == {0: 15.0, 1: 15.0}


def test_single_process_reduction_is_identity():
    assert not dist.is_initialized()
    assert bench.max_over_ranks(3.25) == 3.25


def test_job_throughput_is_weak_scaling():
    # two ranks, each 1 TFLOP in 1 ms -> 2 TFLOP per 1 ms = 2000 TFLOP/s
    assert bench.job_tflops(1e12, 2, 1.0) == pytest.approx(2000.0)
    assert bench.job_tflops(1e12, 1, 2.0) == pytest.approx(500.0)


def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--workload", "b1_h2_n256_d64"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    # the keys of the bench line contract
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["steps"] == 1 and line["warmup"] == 3 and line["higher_is_better"] is True
    assert line["config"]["workload"] == "b1_h2_n256_d64"
    for key in ("value", "unit", "cores", "kind", "sample"):
        assert key in line["cpu_baseline"], key
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["value"] == line["value"] and line["e2e"]["unit"] == line["unit"]
    assert line["e2e"]["d2h_bytes_per_step"] == 0
