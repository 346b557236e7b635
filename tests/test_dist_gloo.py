"""The multi-process side of bench.py on CPU: two ranks over gloo (the GPU
run uses the same code over nccl, one rank per GPU, each an independent
replica -- the decode path has no collective).  Checks the barrier, the
max-over-ranks time and the summed work the weak-scaling value is built from,
and that only rank 0 runs and prints the reference arm."""
from __future__ import annotations

import json
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist(0)
    d.barrier()
    slowest = d.max(1.5 + rank)          # per-rank elapsed ms -> the job's time
    tokens = d.sum(1024.0 * (rank + 1))  # per-rank work -> the job's work
    d.barrier()
    q.put((rank, d.world, slowest, tokens))
    d.pg.destroy_process_group()


def test_bench_dist_two_ranks_over_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2, 2.5, 3072.0), (1, 2, 2.5, 3072.0)]


def test_reference_arm_runs_on_rank_zero_only(capsys, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    class FakeDist:
        rank, world, local, pg = 1, 2, 1, None

    called = []
    monkeypatch.setattr(bench, "oracle_tokens_per_s", lambda *a, **k: called.append(a) or (1.0, 1.0))
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"])
    args = bench.parse_args()
    bench.run_reference(args, FakeDist())
    assert called == [] and capsys.readouterr().out == ""
    FakeDist.rank = 0
    bench.run_reference(args, FakeDist())
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["e2e"]["h2d_bytes_per_step"] == 0
