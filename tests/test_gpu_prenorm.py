"""Pre-normed block on the GPU: with a layer's norm_weight set, every decode
path (single token on thread-block clusters, the fused 1..4-token kernel,
the generic kernels) and the grouped prefill compute
out = x + MoE(x * gamma / sqrt(mean(x^2) + eps)).  Compared with the oracle's
pre-normed block under the same rules as the plain block (tests/parity.py).
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from quantized_moe_expert_gemv_gb300 import binding, build, device, synth
from tests import parity
from tests.test_gpu_prefill import run_prefill

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    binding.load_library()
    oracle.build()


def prenorm_layer(shape, seed, eps=1e-6, bias=None):
    layer = synth.make_layer(shape, seed=seed, router_bias=bias)
    layer.norm_weight = synth.make_norm_weight(shape, seed=seed)
    layer.norm_eps = eps
    return layer


def decode(layer, x_bits, plan=None, scratch=None, dl=None):
    s = layer.shape
    n = x_bits.shape[0]
    dl = dl or device.to_device(layer)
    plan = plan or binding.si_moe_plan(device.desc_for(s))
    scratch = scratch if scratch is not None else device.alloc_scratch(plan, binding.SI_MODE_DECODE, n)
    x = device.tokens_to_device(x_bits)
    out = torch.full((n, s.hidden), float("nan"), dtype=torch.float32, device="cuda")
    ids = torch.full((n, s.top_k), -1, dtype=torch.int32, device="cuda")
    w = torch.empty((n, s.top_k), dtype=torch.float32, device="cuda")
    counts = torch.full((s.n_experts,), -1, dtype=torch.int32, device="cuda")
    logits = torch.empty((n, s.n_experts), dtype=torch.float32, device="cuda")
    ro = binding.route_struct(topk_ids=ids, topk_w=w, expert_counts=counts, logits=logits)
    binding.si_moe_forward_decode(plan, dl.struct(), x, n, out, ro, scratch)
    assert binding.si_moe_read_status(plan, scratch) == binding.SI_OK
    return dict(out=out.cpu().numpy(), ids=ids.cpu().numpy(), w=w.cpu().numpy(),
                counts=counts.cpu().numpy(), logits=logits.cpu().numpy())


def check(layer, x_bits, r, sample=None, max_near=0):
    s = layer.shape
    T = x_bits.shape[0]
    o_ids, o_w, z64, margin = oracle.route_tokens_prenorm(layer.router_w, x_bits, s.top_k, layer.norm_weight,
                                                          layer.norm_eps, bias=layer.router_bias)
    zerr = float(np.max(np.abs(r["logits"].astype(np.float64) - z64)))
    assert zerr <= 0.5 * parity.TAU, f"router logits of the normalised rows off by {zerr:.2e}"
    near = 0
    for t in range(T):
        if not parity.routing_ok(r["ids"][t], o_ids[t], z64[t], margin[t], s.top_k):
            near += 1
            continue
        parity.same_by_id(r["ids"][t], r["w"][t], o_ids[t], o_w[t], atol=2e-6)
    assert near <= max_near, f"{near} near-tie tokens of {T}"
    for t in (range(T) if sample is None else sample):
        if set(r["ids"][t].tolist()) != set(o_ids[t].tolist()):
            continue
        ref = oracle.moe_token_prenorm(layer, x_bits[t], layer.norm_weight, layer.norm_eps)
        parity.assert_close(r["out"][t], ref.out64, f"pre-normed token {t}")
    assert np.isfinite(r["out"]).all()


def test_prenorm_decode_single_token_qwen3_layer():
    wl = synth.WORKLOADS["layer"]
    shape = wl["shape"]
    layer = prenorm_layer(shape, seed=wl["seed"])
    dl = device.to_device(layer)
    plan = binding.si_moe_plan(device.desc_for(shape))
    assert binding.si_debug_decode_fused(plan, 1) == 2  # the cluster kernel
    scratch = device.alloc_scratch(plan, binding.SI_MODE_DECODE, 1)
    xs = synth.make_tokens(shape, seed=41, n_tokens=6)
    for t in range(6):
        r = decode(layer, xs[t:t + 1], plan, scratch, dl)
        assert np.array_equal(r["counts"], np.bincount(r["ids"][0], minlength=shape.n_experts))
        check(layer, xs[t:t + 1], r)


@pytest.mark.parametrize("n", [2, 4])
def test_prenorm_decode_dedup_batches(n):
    wl = synth.WORKLOADS["dedup4"]
    shape, seed = wl["shape"], wl["seed"]
    layer = prenorm_layer(shape, seed=seed, bias=synth.dedup_router_bias(seed, synth.load_dedup_beta()))
    dl = device.to_device(layer)
    plan = binding.si_moe_plan(device.desc_for(shape))
    scratch = device.alloc_scratch(plan, binding.SI_MODE_DECODE, n)
    x = synth.make_tokens(shape, seed=42, n_tokens=2 * n)
    for step in range(2):
        xb = x[n * step: n * (step + 1)]
        r = decode(layer, xb, plan, scratch, dl)
        check(layer, xb, r)


@pytest.mark.parametrize("H,I,E,k,n", [
    (256, 256, 8, 2, 1),     # tiny: cluster kernel
    (1024, 256, 32, 1, 4),   # fused kernel, four tokens
    (768, 512, 4, 4, 2),     # three blocks per row: generic kernels
    (4096, 256, 8, 8, 2),    # sixteen blocks per row: generic kernels
])
def test_prenorm_decode_shapes(H, I, E, k, n):
    shape = synth.MoeShape(H, I, E, k)
    layer = prenorm_layer(shape, seed=H + I + E + k + 1, eps=1e-5)
    x = synth.make_tokens(shape, seed=43, n_tokens=n)
    check(layer, x, decode(layer, x))


def test_prenorm_decode_zero_experts_return_the_input():
    shape = synth.MoeShape(512, 256, 8, 2)
    layer = prenorm_layer(shape, seed=44)
    for name in ("w_gate", "w_up", "w_down"):
        getattr(layer, name)[:] = 0
    for n in (1, 3):
        x = synth.make_tokens(shape, seed=44 + n, n_tokens=n)
        r = decode(layer, x)
        assert np.array_equal(r["out"], synth.bf16_to_f32(x))


def test_prenorm_prefill_shapes():
    for (H, I, E, k, T) in ((256, 256, 8, 2, 37), (512, 512, 40, 6, 300)):
        shape = synth.MoeShape(H, I, E, k)
        layer = prenorm_layer(shape, seed=H + E + T)
        x = synth.make_tokens(shape, seed=T, n_tokens=T)
        r = run_prefill(layer, x)
        g = np.random.default_rng(T)
        sample = sorted(set(g.choice(T, size=min(T, 16), replace=False).tolist()) | {0, T - 1})
        check(layer, x, r, sample, max_near=max(2, T // 100))


def test_prenorm_prefill_qwen3_workload_sampled():
    wl = synth.WORKLOADS["prefill"]
    shape, T = wl["shape"], wl["n_tokens"]
    layer = prenorm_layer(shape, seed=wl["seed"])
    x = synth.make_tokens(shape, seed=wl["seed"], n_tokens=T)
    r = run_prefill(layer, x)
    g = np.random.default_rng(8)
    sample = sorted(set(g.choice(T, size=12, replace=False).tolist()) | {0, T - 1})
    check(layer, x, r, sample, max_near=T // 100)


def test_prenorm_argument_errors():
    shape = synth.TINY
    layer = prenorm_layer(shape, seed=0)
    dl = device.to_device(layer)
    plan = binding.si_moe_plan(device.desc_for(shape))
    scratch = device.alloc_scratch(plan, binding.SI_MODE_DECODE, 1)
    x = device.tokens_to_device(synth.make_tokens(shape, seed=1, n_tokens=1))
    out = torch.empty((1, shape.hidden), dtype=torch.float32, device="cuda")
    bad = dl.struct()
    bad.norm_eps = -1.0
    st = binding.si_moe_forward_decode(plan, bad, x, 1, out, None, scratch, raw_status=True)
    assert st == binding.SI_ERR_INVALID_ARG
    bad = dl.struct()
    bad.norm_eps = float("nan")
    st = binding.si_moe_forward_decode(plan, bad, x, 1, out, None, scratch, raw_status=True)
    assert st == binding.SI_ERR_INVALID_ARG
    gam = torch.zeros(shape.hidden + 1, dtype=torch.float32, device="cuda")
    bad = binding.layer_struct(dl.w_gate, dl.w_up, dl.w_down, dl.router_w, None, gam[1:], 1e-6)
    st = binding.si_moe_forward_decode(plan, bad, x, 1, out, None, scratch, raw_status=True)
    assert st == binding.SI_ERR_MISALIGNED
    assert binding.si_moe_read_status(plan, scratch) == binding.SI_OK
