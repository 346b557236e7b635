"""Parity sample of the 48-layer stack workload's own inputs.

The stack (16 GB of Q4_K experts) is drawn on the device by torch's CUDA
generator (synth.make_layer_torch / make_tokens_torch), not by the numpy
generator the other parity tests use.  This test draws two of its layers
(the first and the last) and the stack's tokens exactly as the benchmark
does, runs the same launch configuration (one CUDA graph of sequential
single-token decode calls, layer after layer), copies those layers' bytes
and the outputs back, and checks sampled (step, layer) tokens against the
CPU oracle under the usual parity rules.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
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
    oracle.build()


def test_stack48_layers_and_tokens_sampled_against_oracle():
    wl = synth.WORKLOADS["stack48"]
    shape, seed, NL, S = wl["shape"], wl["seed"], wl["n_layers"], wl["n_steps"]
    layer_ids = [0, NL - 1]
    steps = [0, 1, S - 1]
    layers = {l: synth.make_layer_torch(shape, seed, l) for l in layer_ids}
    x = synth.make_tokens_torch(S * NL, shape.hidden, (seed, "stack-x")).view(S, NL, shape.hidden)
    plan = binding.si_moe_plan(device.desc_for(shape))
    scratch = device.alloc_scratch(plan, binding.SI_MODE_DECODE, 1)
    structs = {l: binding.layer_struct(*layers[l]) for l in layer_ids}
    calls = [(s, l) for s in steps for l in layer_ids]
    out = torch.full((len(calls), shape.hidden), float("nan"), dtype=torch.float32, device="cuda")
    ids = torch.full((len(calls), shape.top_k), -1, dtype=torch.int32, device="cuda")
    routes = [binding.route_struct(topk_ids=ids[i]) for i in range(len(calls))]
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for i, (s, l) in enumerate(calls):
                binding.si_moe_forward_decode(plan, structs[l], x[s, l], 1, out[i], routes[i], scratch,
                                              stream=stream)
    g.replay()
    assert binding.si_moe_read_status(plan, scratch, stream) == binding.SI_OK
    got, gids = out.cpu().numpy(), ids.cpu().numpy()
    xb = x.view(torch.int16).cpu().numpy().view(np.uint16)
    checked = 0
    for l in layer_ids:
        wg, wu, wd, rw = layers[l]
        host = synth.MoeLayer(shape, wg.cpu().numpy(), wu.cpu().numpy(), wd.cpu().numpy(), rw.cpu().numpy())
        for i, (s, ll) in enumerate(calls):
            if ll != l:
                continue
            o_ids, o_w, z64, margin = oracle.route_tokens(host.router_w, xb[s, l][None], shape.top_k,
                                                          want_logits=True)
            if not parity.routing_ok(gids[i], o_ids[0], z64[0], margin[0], shape.top_k):
                continue
            ref = oracle.moe_token(host, xb[s, l])
            parity.assert_close(got[i], ref.out64, f"stack step {s} layer {l}")
            checked += 1
    assert checked >= len(calls) - 1
