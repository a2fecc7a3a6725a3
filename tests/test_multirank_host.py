"""Multi-rank host logic of bench.py on CPU (gloo, world_size 2).

Every rank runs the whole producer step on its own rows (replicas: the rows
of the producers shard with no exchange), so the only cross-rank steps are a
barrier and the max over ranks of the elapsed time; the reported value is the
bytes all ranks moved over that time.  The reference arm (the CPU oracle) runs
on rank 0 only and the other ranks exit 0 without output.
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


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(5.0 + 2.0 * rank, world, torch.device("cpu"))
        dist.barrier()
        out.put((rank, ms, bench.job_gbs(1_000_000, world, ms)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    mp.start_processes(_worker, args=(world, _free_port(), q), nprocs=world, join=True, start_method="spawn")
    res = sorted(q.get() for _ in range(world))
    for rank, ms, gbs in res:
        assert ms == 7.0                              # the slower rank's time, on every rank
        assert gbs == pytest.approx(2 * 1_000_000 / 7e-3 / 1e9)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.job_gbs(7_000_000, 1, 1.0) == pytest.approx(7.0)


def _reference(rank: int, world: int):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
               MASTER_ADDR="127.0.0.1", MASTER_PORT="29999")
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_other_ranks_exit_quietly():
    r = _reference(1, 2)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_reference_arm_rank0_prints_one_line():
    r = _reference(0, 2)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "GB/s"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
