"""The N > 1 host path of bench.py on CPU: world-size-2 gloo process groups.

The forward linear layer shards over tokens with no exchange, so
`bench.py --gpus N` runs N replicas ("replicas only", weak scaling): each
rank times its own replica, the ranks agree on the slowest time by an
all-reduce, and the whole-job value is every rank's FLOPs over that time.
The reference arm runs on rank 0 alone. No GPU is used.
"""

import io
import json
import os
import socket
import subprocess
import sys
from contextlib import redirect_stdout

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            init_method=f"tcp://127.0.0.1:{port}")
    try:
        ms_max = bench.max_over_ranks(times[rank], dist, "cpu")
        value = bench.replicas_value(world, 2.0e12, ms_max)
        dist.barrier()
        q.put((rank, ms_max, value))
    finally:
        dist.destroy_process_group()


def _run(times):
    world = len(times)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(out)


def test_ranks_agree_on_the_slowest_time():
    out = _run([2.0, 3.5])
    assert [r for r, _, _ in out] == [0, 1]
    for _, ms_max, value in out:
        assert ms_max == 3.5
        # two replicas of 2 TFLOP each in 3.5 ms
        assert abs(value - 2 * 2.0e12 / 3.5e-3 / 1e12) < 1e-9


def test_single_rank_is_the_identity():
    import bench
    assert bench.max_over_ranks(1.25, None, "cpu") == 1.25
    assert abs(bench.replicas_value(1, 1.0e12, 1.0) - 1000.0) < 1e-9


def test_reference_arm_runs_on_rank_0_only():
    import argparse

    import bench
    args = argparse.Namespace(workload=bench.HEADLINE, warmup=3, steps=1, ref_rows=1)
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(args, rank=1) is None
    assert buf.getvalue() == ""


def test_gpus_flag_starts_the_ranks():
    # `bench.py --gpus 2` with no launcher around it starts two ranks itself
    # (torch.distributed.run on 127.0.0.1); the reference arm then runs on
    # rank 0, which prints the one JSON line, and rank 1 says it has no work.
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    env["OMP_NUM_THREADS"] = "2"
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2",
                        "--impl", "reference", "--workload", "attn_proj_f32", "--steps", "1",
                        "--warmup", "3", "--ref-rows", "2"],
                       cwd=ROOT, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["config"]["workload"] == "attn_proj_f32"
    assert "rank 1 of 2: the reference arm runs on rank 0 only" in r.stderr
