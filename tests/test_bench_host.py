"""Host-side logic of bench.py that needs no GPU, run against fakes of the
CUDA pieces: the per-token end-to-end loop (one copy in, one decode call, one
copy out and one wait per token) and the figures it reports."""
from __future__ import annotations

import contextlib
import os
import sys
import types

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


class _T:
    def __init__(self, shape, log, name):
        self.shape, self.log, self.name = tuple(shape), log, name

    def pin_memory(self):
        return self

    def __getitem__(self, i):
        assert 0 <= i < self.shape[0]
        return _T(self.shape[1:], self.log, f"{self.name}[{i}]")

    def copy_(self, src, non_blocking=False):
        assert non_blocking and src.shape == self.shape
        self.log.append(("copy", self.name, src.name))
        return self


def _fakes(log):
    class Stream:
        def synchronize(self):
            log.append(("sync",))

    torch = types.SimpleNamespace(
        int16="int16", float32="float32",
        empty=lambda shape, dtype=None, device=None: _T(shape, log, f"{device or 'host'}:{dtype}"),
        cuda=types.SimpleNamespace(stream=lambda s: contextlib.nullcontext(), synchronize=lambda: None))
    binding = types.SimpleNamespace(
        SI_OK=0, si_status_string=str, si_moe_read_status=lambda plan, scratch, stream: 0,
        si_moe_forward_decode=lambda plan, L, x, n, out, ro, scratch, stream=None:
            log.append(("decode", x.name, n, out.name)))
    dist = types.SimpleNamespace(barrier=lambda: None, max=lambda v: v, sum=lambda v: v)
    return torch, binding, dist, Stream()


def test_e2e_per_token_copies_calls_and_waits_once_per_token():
    sys.path.insert(0, ROOT)
    import bench
    log = []
    torch, binding, dist, stream = _fakes(log)
    shape = types.SimpleNamespace(hidden=2048)
    x_pin = _T((8, 2048), log, "x_pin")
    r = bench.e2e_per_token(binding, "plan", "L", x_pin, "scratch", stream, shape, dist, torch, n=5, warmup=3)
    per_token = [("copy", "cuda:int16", None), ("decode", "cuda:int16", 1, "cuda:float32"),
                 ("copy", None, "cuda:float32"), ("sync",)]
    assert len(log) == 4 * (3 + 5)
    for i, t in enumerate(list(range(3)) + list(range(5))):  # warm-up tokens, then the timed ones
        got = log[4 * i: 4 * i + 4]
        assert [g[0] for g in got] == [p[0] for p in per_token]
        assert got[0][2] == f"x_pin[{t}]" and got[1][1:] == per_token[1][1:]
        assert got[2][1] == f"host:float32[{t}]"
    assert r["tokens"] == 5 and r["unit"] == "tok/s" and r["value"] > 0
    assert r["h2d_bytes_per_token"] == 2048 * 2 and r["d2h_bytes_per_token"] == 2048 * 4
    assert abs(r["us_per_token"] * r["value"] - 1e6) < 1e-6 * 1e6
