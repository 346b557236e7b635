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
        SI_MODE_DECODE_HOST=2,
        si_moe_forward_decode=lambda plan, L, x, n, out, ro, scratch, stream=None:
            log.append(("decode", x.name, n, out.name)),
        si_moe_forward_decode_host=lambda plan, L, x, n, out, ro, scratch, stream=None:
            log.append(("decode_host", x.name, n, out.name, scratch)))
    dist = types.SimpleNamespace(barrier=lambda: None, max=lambda v: v, sum=lambda v: v)
    device = types.SimpleNamespace(alloc_scratch=lambda plan, mode, n: f"scratch(mode={mode}, n={n})")
    return torch, binding, dist, device, Stream()


def test_e2e_per_token_copies_calls_and_waits_once_per_token():
    sys.path.insert(0, ROOT)
    import bench
    log = []
    torch, binding, dist, device, stream = _fakes(log)
    shape = types.SimpleNamespace(hidden=2048)
    x_pin = _T((8, 2048), log, "x_pin")
    r = bench.e2e_per_token(binding, device, "plan", "L", x_pin, "scratch", stream, shape, dist, torch,
                            n=5, warmup=3)
    order = list(range(3)) + list(range(5))  # warm-up tokens, then the timed ones
    # the host-buffer entry point: one call per token, its own scratch
    host = log[:len(order)]
    assert host == [("decode_host", f"x_pin[{t}]", 1, f"host:float32[{t}]", "scratch(mode=2, n=1)")
                    for t in order]
    # torch's copies around the device entry point: copy in, decode, copy out, wait
    rest = log[len(order):]
    assert len(rest) == 4 * len(order)
    for i, t in enumerate(order):
        got = rest[4 * i: 4 * i + 4]
        assert got == [("copy", "cuda:int16", f"x_pin[{t}]"), ("decode", "cuda:int16", 1, "cuda:float32"),
                       ("copy", f"host:float32[{t}]", "cuda:float32"), ("sync",)]
    assert r["tokens"] == 5 and r["unit"] == "tok/s" and r["value"] > 0 and r["torch_copies"]["value"] > 0
    assert r["h2d_bytes_per_token"] == 2048 * 2 and r["d2h_bytes_per_token"] == 2048 * 4
    assert abs(r["us_per_token"] * r["value"] - 1e6) < 1.0
