"""Multi-process (gloo, world size 2, CPU) checks of the benchmark's rank
logic: every rank runs an independent replica of the step, the job's time
is the slowest rank's, ``value`` counts every rank's work, and only rank 0
reports.  Nothing here needs a GPU."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    r, w, local = bench.dist_init(world)
    assert (r, w, local) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    t_local = 10.0 + 5.0 * rank          # ms of this rank's timed region
    t_max = bench.max_over_ranks(t_local, w)
    bench.barrier(w)
    v = bench.aggregate_value(bench.STEP_FLOPS, 4, w, t_max)
    q.put((rank, t_max, v))
    dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_gloo_world2():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for pr in procs:
        pr.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    import bench
    for rank, t_max, v in res:
        assert t_max == 15.0                          # the slowest rank's time
        assert v == pytest.approx(bench.STEP_FLOPS * 4 * 2 / 15e-3 / 1e12)


def test_reference_arm_only_rank0_reports():
    """Under torchrun the reference arm runs on rank 0 only; other ranks exit 0 silently."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0"], capture_output=True, text=True, env=env,
                         timeout=300)
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_reference_arm_rank0_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0"], capture_output=True, text=True, env=env,
                         timeout=600)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "TFLOP/s"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_bench_modes_present():
    """Every bench mode the design notes cite exists and is wired to its flag."""
    sys.path.insert(0, ROOT)
    import bench
    for name in ("run_ours", "run_reference", "run_configs", "run_sweep", "profile_case", "workloads",
                 "cpu_baseline", "aggregate_value", "run_precision_report", "run_trace", "profile_workload"):
        assert callable(getattr(bench, name)), name
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--help"], capture_output=True,
                         text=True, timeout=120)
    for flag in ("--configs", "--sweep", "--profile-case", "--tile-mode", "--impl", "--gpus", "--steps", "--warmup",
                 "--precision-report", "--trace", "--profile-workload"):
        assert flag in out.stdout, flag
