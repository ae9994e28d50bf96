"""The N>1 path of bench.py on CPU, with the gloo backend and two ranks.

bench.py runs N independent replicas (one process per GPU, no collective on the data
path). Across ranks it only agrees on time: the job's step time is the slowest
replica's, and the job's throughput counts every replica's work. These tests run that
logic with two gloo ranks, and the reference arm under torchrun, where rank 0 alone
does the work and prints the line.
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


def _rank_main(rank: int, world: int, port: int, local_ms: list, out_q):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        ms = bench.max_over_ranks(local_ms[rank], "cpu")
        out_q.put((rank, ms, bench.job_throughput(1000.0, world, ms)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    local_ms = [2.5, 4.0]  # rank 1 is the slower replica
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, local_ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # Both ranks agree on the slowest time; throughput = 2 replicas x 1000 units / 4 ms.
    assert [g[1] for g in got] == [4.0, 4.0]
    assert all(abs(g[2] - 2 * 1000.0 / 4e-3) < 1e-6 for g in got)


def test_single_process_helpers_without_a_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.25, "cpu") == 3.25
    assert bench.job_throughput(500.0, 1, 2.0) == pytest.approx(250000.0)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_zero():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "mha_tiny"]
    env = {**os.environ, "CUDA_VISIBLE_DEVICES": "", "OMP_NUM_THREADS": "1"}
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["unit"] == "GB/s"
    assert line["e2e"]["value"] == line["value"]


@pytest.mark.parametrize("workload,metric,unit", [
    ("mla_spec", "MLA absorbed paged decode: achieved HBM GB/s and TFLOP/s", "GB/s"),
    ("mixed_prefill", "causal paged prefill (mixed with decode rows): achieved TFLOP/s", "TFLOP/s"),
    ("scatter", "kv_cache_write scatter: achieved HBM GB/s", "GB/s"),
    ("mla_write", "fused MLA RMSNorm+RoPE cache write: achieved HBM GB/s", "GB/s"),
])
def test_reference_arm_times_the_oracle_on_the_workloads_own_metric(workload, metric, unit):
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--workload", workload, "--steps", "1",
           "--warmup", "0", "--ref-budget-s", "1"]
    if workload in ("scatter", "mla_write"):
        cmd += ["--batch", "8192"]
    env = {**os.environ, "CUDA_VISIBLE_DEVICES": "", "OMP_NUM_THREADS": "1"}
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])
    assert line["impl"] == "reference" and line["metric"] == metric and line["unit"] == unit
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["value"] == line["value"]


def test_reference_arm_without_an_oracle_leg_says_so():
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--workload", "fork"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300,
                       env={**os.environ, "CUDA_VISIBLE_DEVICES": ""})
    assert r.returncode == 0
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and "unavailable" in line
