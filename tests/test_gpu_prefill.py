"""GPU parity of the grouped prefill (routing, counts/offsets/perm, CTA-pair
tensor-core gate/up and down GEMMs on fp16-dequantized Q4_K operands,
slot-order combine) against the CPU oracle, through the C ABI."""
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


def run_prefill(layer: synth.MoeLayer, x_bits: np.ndarray, max_tokens=None, dl=None):
    s = layer.shape
    T = x_bits.shape[0]
    dl = dl or device.to_device(layer)
    plan = binding.si_moe_plan(binding.make_desc(s.hidden, s.intermediate, s.n_experts, s.top_k,
                                                 max_tokens=max_tokens or T))
    scratch = device.alloc_scratch(plan, binding.SI_MODE_PREFILL, T)
    x = device.tokens_to_device(x_bits)
    out = torch.full((T, s.hidden), float("nan"), dtype=torch.float32, device="cuda")
    ids = torch.full((T, s.top_k), -1, dtype=torch.int32, device="cuda")
    w = torch.empty((T, s.top_k), dtype=torch.float32, device="cuda")
    counts = torch.full((s.n_experts,), -1, dtype=torch.int32, device="cuda")
    offsets = torch.full((s.n_experts + 1,), -1, dtype=torch.int32, device="cuda")
    perm = torch.full((T * s.top_k,), -1, dtype=torch.int32, device="cuda")
    logits = torch.empty((T, s.n_experts), dtype=torch.float32, device="cuda")
    ro = binding.route_struct(topk_ids=ids, topk_w=w, expert_counts=counts, expert_offsets=offsets,
                              perm=perm, logits=logits)
    binding.si_moe_forward_prefill(plan, dl.struct(), x, T, out, ro, scratch)
    assert binding.si_moe_read_status(plan, scratch) == binding.SI_OK
    return dict(out=out.cpu().numpy(), ids=ids.cpu().numpy(), w=w.cpu().numpy(), counts=counts.cpu().numpy(),
                offsets=offsets.cpu().numpy(), perm=perm.cpu().numpy(), logits=logits.cpu().numpy())


def check_prefill(layer, x_bits, r, sample):
    s = layer.shape
    T = x_bits.shape[0]
    # routing against the oracle (fp32 decisions, margin rule)
    o_ids, o_w, z64, margin = oracle.route_tokens(layer.router_w, x_bits, s.top_k, bias=layer.router_bias,
                                                  want_logits=True)
    near = 0
    for t in range(T):
        if not parity.routing_ok(r["ids"][t], o_ids[t], z64[t], margin[t], s.top_k):
            near += 1
            continue
        parity.same_by_id(r["ids"][t], r["w"][t], o_ids[t], o_w[t], atol=2e-6)
    assert near <= max(2, T // 100), f"{near} near-tie tokens of {T}"
    # fp32 logits within half the tie threshold of the fp64 ones (so every token whose
    # fp64 margin is >= the threshold is decided identically on both sides)
    zerr = float(np.max(np.abs(r["logits"].astype(np.float64) - z64)))
    assert zerr <= 0.5 * parity.TAU, f"router logits off by {zerr:.2e}"
    # same fp32 logits -> the same selection, bit for bit
    for t in range(0, T, max(1, T // 64)):
        assert np.array_equal(r["ids"][t], oracle.topk(r["logits"][t], s.top_k))
    # bookkeeping on the GPU's own ids: bit-exact
    counts, offsets, perm = oracle.counts_offsets_perm(r["ids"], s.n_experts)
    assert np.array_equal(r["counts"], counts)
    assert np.array_equal(r["offsets"], offsets)
    assert np.array_equal(r["perm"], perm)
    # outputs of sampled tokens (whose selection matches the oracle's)
    checked = 0
    for t in sample:
        if set(r["ids"][t].tolist()) != set(o_ids[t].tolist()):
            continue
        ref = oracle.moe_token(layer, x_bits[t])
        parity.assert_close(r["out"][t], ref.out64, f"prefill token {t}")
        checked += 1
    assert checked >= len(sample) // 2
    assert np.isfinite(r["out"]).all()


def test_prefill_tiny_layer_ragged():
    layer = synth.make_layer(synth.TINY, seed=0)
    x = synth.make_tokens(synth.TINY, seed=0, n_tokens=37)
    r = run_prefill(layer, x)
    check_prefill(layer, x, r, range(37))


def test_prefill_single_token():
    layer = synth.make_layer(synth.TINY, seed=0)
    x = synth.make_tokens(synth.TINY, seed=5, n_tokens=1)
    r = run_prefill(layer, x, max_tokens=64)
    check_prefill(layer, x, r, [0])


@pytest.mark.parametrize("H,I,E,k,T", [
    (256, 512, 8, 2, 2100),    # experts with > 512 pairs: several passes per tile
    (512, 256, 16, 4, 300),    # two blocks per gate row, one per down row
    (768, 768, 6, 3, 129),     # three blocks each way, ragged tiles
    (256, 256, 1, 1, 70),      # one expert
    (256, 256, 160, 16, 96),   # two router expert passes (128 + 32), top-16
    (512, 512, 40, 6, 777),    # ragged token chunks, one- and two-chunk passes
])
def test_prefill_shapes(H, I, E, k, T):
    shape = synth.MoeShape(H, I, E, k)
    layer = synth.make_layer(shape, seed=H + I + E + k)
    x = synth.make_tokens(shape, seed=T, n_tokens=T)
    r = run_prefill(layer, x)
    g = np.random.default_rng(T)
    sample = sorted(set(g.choice(T, size=min(T, 24), replace=False).tolist()) | {0, T - 1})
    check_prefill(layer, x, r, sample)


def test_prefill_qwen3_workload_sampled():
    wl = synth.WORKLOADS["prefill"]
    shape, T = wl["shape"], wl["n_tokens"]
    layer = synth.make_layer(shape, seed=wl["seed"])
    x = synth.make_tokens(shape, seed=wl["seed"], n_tokens=T)
    r = run_prefill(layer, x)
    g = np.random.default_rng(7)
    sample = sorted(set(g.choice(T, size=24, replace=False).tolist()) | {0, T - 1})
    check_prefill(layer, x, r, sample)


def test_prefill_argument_errors():
    layer = synth.make_layer(synth.TINY, seed=0)
    s = layer.shape
    dl = device.to_device(layer)
    plan = binding.si_moe_plan(binding.make_desc(s.hidden, s.intermediate, s.n_experts, s.top_k, max_tokens=16))
    scratch = device.alloc_scratch(plan, binding.SI_MODE_PREFILL, 16)
    x = device.tokens_to_device(synth.make_tokens(s, seed=1, n_tokens=16))
    out = torch.empty((16, s.hidden), dtype=torch.float32, device="cuda")
    st = binding.si_moe_forward_prefill(plan, dl.struct(), x, 0, out, None, scratch, raw_status=True)
    assert st == binding.SI_ERR_INVALID_ARG
    st = binding.si_moe_forward_prefill(plan, dl.struct(), x, 17, out, None, scratch, raw_status=True)
    assert st == binding.SI_ERR_INVALID_ARG
    small = scratch[: scratch.numel() // 2]
    st = binding.si_moe_forward_prefill(plan, dl.struct(), x, 16, out, None, small, raw_status=True)
    assert st == binding.SI_ERR_SCRATCH_TOO_SMALL
    st = binding.si_moe_forward_prefill(plan, dl.struct(), x[:, 1:], 16, out, None, scratch, raw_status=True)
    assert st == binding.SI_ERR_MISALIGNED
    assert binding.si_moe_read_status(plan, scratch) == binding.SI_OK
