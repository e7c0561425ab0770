"""The N>1 bench path on CPU ranks (gloo, world size 2).

Each rank serves its own batch and no collective touches the data path; the
job's time is the slowest rank's, and its throughput counts every rank's tokens.
"""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")    # rank 1 is the slow one
        q.put((rank, ms, bench.job_value(16, world, ms)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank_and_all_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, value in got:
        assert ms == 15.0                              # max over ranks, on every rank
        assert abs(value - 2 * 16 / 15e-3) < 1e-6      # both ranks' tokens over the job's time


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_value(16, 1, 2.0) == 8000.0


def _reference(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--workload", "prefill_4k", "--steps", "1", "--warmup", "0", "--gpus", "2"],
                          capture_output=True, text=True, env=env, timeout=600)


def test_reference_arm_under_two_ranks():
    r1 = _reference(1)                                 # other ranks exit without work
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = _reference(0)                                 # rank 0 prints the one line
    assert r0.returncode == 0, r0.stderr
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
