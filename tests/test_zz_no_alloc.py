"""The decode entry point for callers that cannot allocate device memory.

A plug-in living inside a host framework whose memory pool owns all device
memory, or a latency-critical decode loop that must not call cudaMalloc
(which synchronises the device), cannot hand the library a scratch buffer.
si_moe_forward_decode_noalloc serves them with a fixed device array built
into the library.  This test calls it twice in a row through the C ABI and
checks each result against the regular entry point with a caller-owned
scratch buffer, at the same tolerance as the other parity tests.  It lives in
a file of its own that pytest collects last, and passes both alone in a fresh
process and after the rest of the suite.
"""
from __future__ import annotations

import numpy as np
import pytest

from quantized_moe_expert_gemv_gb300 import binding, build, device, synth
from tests import parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    binding.load_library()


def test_noalloc_decode_matches_caller_scratch_decode_on_two_calls_in_a_row():
    shape = synth.QWEN3_30B_A3B
    layer = synth.make_layer(shape, seed=1)
    dl = device.to_device(layer)
    L = dl.struct()
    plan = binding.si_moe_plan(device.desc_for(shape))
    scratch = device.alloc_scratch(plan, binding.SI_MODE_DECODE, binding.SI_MAX_DECODE_TOKENS)
    calls = [synth.make_tokens(shape, seed=41, n_tokens=1),
             synth.make_tokens(shape, seed=42, n_tokens=binding.SI_MAX_DECODE_TOKENS)]

    def run(x_bits, noalloc):
        n = x_bits.shape[0]
        x = device.tokens_to_device(x_bits)
        out = torch.full((n, shape.hidden), float("nan"), dtype=torch.float32, device="cuda")
        ids = torch.full((n, shape.top_k), -1, dtype=torch.int32, device="cuda")
        ro = binding.route_struct(topk_ids=ids)
        if noalloc:
            binding.si_moe_forward_decode_noalloc(plan, L, x, n, out, ro)
        else:
            binding.si_moe_forward_decode(plan, L, x, n, out, ro, scratch)
        return out, ids

    # two no-allocation calls back to back, then the reference calls
    got = [run(x, noalloc=True) for x in calls]
    torch.cuda.synchronize()
    want = [run(x, noalloc=False) for x in calls]
    torch.cuda.synchronize()
    for (o, i), (ro_, ri) in zip(got, want):
        assert torch.equal(i, ri)
        o_h, r_h = o.cpu().numpy(), ro_.cpu().numpy()
        assert np.isfinite(o_h).all()
        for t in range(o_h.shape[0]):
            parity.assert_close(o_h[t], r_h[t], "no-allocation decode vs caller-scratch decode")
    # no device-side error was recorded in the fixed array, and reading clears nothing else
    assert binding.si_moe_read_status_noalloc() == binding.SI_OK
    assert binding.si_moe_read_status(plan, scratch) == binding.SI_OK


def test_noalloc_decode_rejects_bad_arguments():
    shape = synth.TINY
    dl = device.to_device(synth.make_layer(shape, seed=0))
    plan = binding.si_moe_plan(device.desc_for(shape))
    x = device.tokens_to_device(synth.make_tokens(shape, seed=0, n_tokens=1))
    out = torch.empty((1, shape.hidden), dtype=torch.float32, device="cuda")
    st = binding.si_moe_forward_decode_noalloc(plan, dl.struct(), x, 0, out, raw_status=True)
    assert st == binding.SI_ERR_INVALID_ARG
    st = binding.si_moe_forward_decode_noalloc(plan, dl.struct(), x, 1, out[:, 1:], raw_status=True)
    assert st == binding.SI_ERR_MISALIGNED
    st = binding.si_moe_forward_decode_noalloc(plan, dl.struct(), x[:, 1:], 1, out, raw_status=True)
    assert st == binding.SI_ERR_MISALIGNED
    assert binding.si_moe_read_status_noalloc() == binding.SI_OK


def test_noalloc_decode_rejects_a_shape_beyond_the_fixed_array():
    """A layer whose decode scratch exceeds SI_STATIC_SCRATCH_BYTES (16 tokens'
    worth of h for intermediate 4096, top-16, 4 tokens: 1 MiB of h alone) is
    refused with SI_ERR_SCRATCH_TOO_SMALL, and nothing is written."""
    shape = synth.MoeShape(hidden=256, intermediate=4096, n_experts=16, top_k=16)
    plan = binding.si_moe_plan(device.desc_for(shape))
    assert binding.si_moe_scratch_bytes(plan, binding.SI_MODE_DECODE, 4) > binding.SI_STATIC_SCRATCH_BYTES
    dl = device.to_device(synth.make_layer(shape, seed=0))
    x = device.tokens_to_device(synth.make_tokens(shape, seed=0, n_tokens=4))
    out = torch.full((4, shape.hidden), float("nan"), dtype=torch.float32, device="cuda")
    st = binding.si_moe_forward_decode_noalloc(plan, dl.struct(), x, 4, out, raw_status=True)
    assert st == binding.SI_ERR_SCRATCH_TOO_SMALL
    torch.cuda.synchronize()
    assert torch.isnan(out).all()
    assert binding.si_moe_read_status_noalloc() == binding.SI_OK
