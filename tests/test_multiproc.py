"""The N > 1 path of bench.py on CPU: world size 2 over gloo.

Every rank runs its own replica of the workload (the forward pass has no
exchange step), so the only cross-rank step is the timing reduction: the job
takes the slowest rank's time, and the whole-job value counts every rank's
steps.  The reference arm runs on rank 0 alone.
"""

from __future__ import annotations

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


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [10.0 + 5.0 * rank, 30.0 - 7.0 * rank]      # rank 1 slower in the first
        got = bench.max_over_ranks(mine, world, dist, "cpu")
        value = bench.whole_job_tflops(world, 8.0e9, 4, got[0])
        out.put((rank, got, value))
    finally:
        dist.destroy_process_group()


def test_timing_reduction_takes_the_slowest_rank():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, got, value in results:
        assert got == [15.0, 30.0]
        # two ranks x 4 steps x 8e9 FLOPs over the slowest rank's 15 ms
        assert abs(value - 2 * 4 * 8.0e9 / 15e-3 / 1e12) < 1e-9


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.0, 2.0], 1) == [1.0, 2.0]


def test_reference_arm_under_two_ranks_prints_one_line():
    env = dict(os.environ, PYTHONPATH=ROOT)
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--workload", "single_head_L128_d64"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
