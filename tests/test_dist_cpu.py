"""The multi-process (replica) path of the benchmark on CPU, world size 2
over gloo: the timing is the max over ranks on every rank, the whole-job
value counts every rank's work, and the reference arm runs on rank 0 only."""

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


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench._dist()
        assert (ws, r, local) == (world, rank, rank)
        per_rank_ms = [2.0, 5.0][rank]
        mx = bench._barrier_max(torch, per_rank_ms, ws)
        out[rank] = (mx, bench.whole_job_value(ws, 1e12, mx))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value():
    import torch.multiprocessing as mp
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == out[1]
    mx, value = out[0]
    assert mx == 5.0                                     # the slowest rank decides
    assert value == pytest.approx(2 * 1e12 / 5e-3 / 1e12)   # both ranks' work


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1",
               MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       timeout=120, env=env, cwd=ROOT)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
