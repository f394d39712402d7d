"""The bench's multi-rank host logic on CPU: two gloo ranks, one process each
(the shape of `torchrun --nproc-per-node 2 bench.py`), with no GPU.

* every rank reads its rank and world size from the launcher's environment;
* the timed region's length is the maximum over ranks, and the whole-job
  rate is the evictions all ranks processed over that time (weak scaling);
* the reference arm runs on rank 0 alone; other ranks exit 0 with no output.
"""

from __future__ import annotations

import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q) -> None:
    import torch
    import torch.distributed as dist
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    r, lr, w = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    try:
        elapsed = 100.0 + 25.0 * rank  # rank 1 is the slower one
        m = bench.max_over_ranks(elapsed, w, torch.device("cpu"))
        value = bench.aggregate(6912 * 10, m / 1e3, w)
        q.put((r, lr, w, m, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_work():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for r, (rank, local_rank, w, m, value) in enumerate(got):
        assert (rank, local_rank, w) == (r, r, world)
        assert m == 125.0                                   # the slower rank's time
        assert value == pytest.approx(6912 * 10 * 2 / 0.125)  # both ranks' evictions


def test_max_over_ranks_is_the_identity_for_one_rank():
    import bench
    assert bench.max_over_ranks(42.5, 1, None) == 42.5


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0"],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0
    assert out.stdout.strip() == ""
