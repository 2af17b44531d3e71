"""The multi-GPU plumbing of bench.py on CPU with two gloo ranks: one process
per rank, a barrier, the timing taken as the maximum over ranks and the
whole-job rate from it (requests are independent, so the ranks share no data
and the step has no collective); the reference arm runs on rank 0 only."""

import argparse
import multiprocessing as mp
import os
import socket

import pytest


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    try:
        import bench
        w, r, _ = bench.dist_setup()
        bench.dist_init(w, "gloo")
        bench.barrier(w)
        elapsed_ms = bench.max_over_ranks(w, 100.0 + 50.0 * r)   # rank r "took" 100 + 50 r ms
        rate = bench.aggregate_rate(w, 40, elapsed_ms / 1e3)
        bench.barrier(w)
        import torch.distributed as dist
        dist.destroy_process_group()
        q.put((r, w, elapsed_ms, rate))
    except Exception as e:  # reported to the parent, which fails the test
        q.put((rank, "error", repr(e), None))


def test_two_gloo_ranks_take_the_slowest_rank_and_the_whole_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    got.sort()
    for r, w, elapsed_ms, rate in got:
        assert w == 2, (r, elapsed_ms)
        assert elapsed_ms == 150.0            # max over ranks
        assert rate == pytest.approx(2 * 40 / 0.150)   # both ranks' steps over that time


def test_reference_arm_runs_on_rank_zero_only():
    import bench
    args = argparse.Namespace(workload="b1", steps=1, warmup=1, gpus=2)
    assert bench.run_reference(args, 2, 1) == 0     # returns at once, no oracle work


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.dist_setup()[0] == int(os.environ.get("WORLD_SIZE", "1"))
    assert bench.max_over_ranks(1, 12.5) == 12.5
    bench.barrier(1)
    assert bench.aggregate_rate(1, 100, 0.5) == 200.0


def test_gpus_flag_starts_the_ranks_itself():
    """`bench.py --gpus 2` without a launcher spawns two ranks (127.0.0.1
    rendezvous); on the reference arm rank 0 alone runs the oracle and
    prints one line whose n_gpus is the real world size, rank 1 exits 0."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    env["PE_REF_BUDGET_S"] = "5"
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2",
                        "--impl", "reference", "--workload", "tiny", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["config"]["parallelism"] == "replicas x2"


def test_gpus_flag_must_match_the_launcher_world_size():
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2",
                        "--impl", "reference", "--workload", "tiny", "--steps", "1"],
                       capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 2
    assert "WORLD_SIZE=1" in r.stderr
