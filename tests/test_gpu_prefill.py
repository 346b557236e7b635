"""GPU parity of the grouped prefill (routing, counts/offsets/perm, CTA-pair
tensor-core gate/up and down GEMMs on fp16-dequantized Q4_K operands,
slot-order combine) against the CPU oracle, through the C ABI."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from quantized_moe_expert_gemv_gb300 import binding, build, device, synth
from tests import parity
from tests.q4k_fixtures import dequant_test_blocks

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


# ------------------------------------------------- the GEMM operand conversion
def _f16_bits(values_f32: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp16 of fp32 values, as uint16 bits."""
    with np.errstate(over="ignore"):  # beyond fp16's range -> inf, as the GPU's conversion gives
        return np.asarray(values_f32, dtype=np.float32).astype(np.float16).view(np.uint16)


def test_prefill_operand_dequant_bit_exact_against_oracle():
    """The grouped prefill's own Q4_K -> fp16 conversion (the device function
    its GEMM dequantization warps run, exported for this test) equals the
    round-to-nearest-even fp16 of the oracle's fp32 weight, bit for bit."""
    blocks = dequant_test_blocks()
    n = blocks.shape[0]
    ref = oracle.q4k_dequant(blocks)
    out = torch.empty(n * 256, dtype=torch.int16, device="cuda")
    binding.si_debug_q4k_dequant_f16(torch.from_numpy(blocks).cuda(), n, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint16)
    finite = np.isfinite(ref)
    assert finite.sum() > 0.99 * ref.size
    assert np.array_equal(got[finite], _f16_bits(ref)[finite])
    # the random blocks of the prefill workload's own layer
    wl = synth.WORKLOADS["prefill"]
    layer_blocks = synth.q4k_random_blocks(synth.rng(wl["seed"], 0, "gate"), 100_000)
    ref = oracle.q4k_dequant(layer_blocks)
    out = torch.empty(ref.size, dtype=torch.int16, device="cuda")
    binding.si_debug_q4k_dequant_f16(torch.from_numpy(layer_blocks).cuda(), layer_blocks.shape[0], out)
    assert np.array_equal(out.cpu().numpy().view(np.uint16), _f16_bits(ref))


def test_prefill_operand_dequant_with_norm_gain_bit_exact():
    """Pre-normed block: the gate/up operand is fp16(fp32(w) * gamma_c), the
    fp32 product of the oracle's fp32 weight and the column's gain, rounded
    to nearest even in fp32 and then in fp16."""
    blocks = dequant_test_blocks()
    n = blocks.shape[0]
    gamma = synth.rng(101, "gain").uniform(0.5, 1.5, n * 256).astype(np.float32)
    gamma[:256] = 1.0  # unit gain: the plain conversion
    gamma[256:512] = np.float32(2.0) ** synth.rng(102).integers(-3, 4, 256)  # powers of two: exact products
    ref = oracle.q4k_dequant(blocks)
    expect = _f16_bits(ref * gamma)  # numpy float32 * float32 rounds once, to nearest even
    out = torch.empty(n * 256, dtype=torch.int16, device="cuda")
    binding.si_debug_q4k_dequant_f16(torch.from_numpy(blocks).cuda(), n, out, gamma=torch.from_numpy(gamma).cuda())
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint16)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], expect[finite])
    assert np.array_equal(got[:256][finite[:256]], _f16_bits(ref[:256])[finite[:256]])


# --------------------------------------------------------------- fp16 range
def _status_after_prefill(layer, x_bits):
    s = layer.shape
    T = x_bits.shape[0]
    dl = device.to_device(layer)
    plan = binding.si_moe_plan(binding.make_desc(s.hidden, s.intermediate, s.n_experts, s.top_k, max_tokens=T))
    scratch = device.alloc_scratch(plan, binding.SI_MODE_PREFILL, T)
    out = torch.empty((T, s.hidden), dtype=torch.float32, device="cuda")
    binding.si_moe_forward_prefill(plan, dl.struct(), device.tokens_to_device(x_bits), T, out, None, scratch)
    return binding.si_moe_read_status(plan, scratch), plan, scratch, dl


def _prefill_again_is_correct(layer, plan, scratch, dl):
    """After an error: re-initialise the scratch, run a normal prefill of the
    tiny layer's tokens and check it against the oracle."""
    s = layer.shape
    T = 8  # within the plan's max_tokens (10)
    x = synth.make_tokens(s, seed=3, n_tokens=T)
    binding.si_moe_scratch_init(plan, scratch)
    out = torch.full((T, s.hidden), float("nan"), dtype=torch.float32, device="cuda")
    ids = torch.full((T, s.top_k), -1, dtype=torch.int32, device="cuda")
    binding.si_moe_forward_prefill(plan, dl.struct(), device.tokens_to_device(x), T, out,
                                   binding.route_struct(topk_ids=ids), scratch)
    assert binding.si_moe_read_status(plan, scratch) == binding.SI_OK
    got, gids = out.cpu().numpy(), ids.cpu().numpy()
    for t in range(T):
        ref = oracle.moe_token(layer, x[t])
        if np.array_equal(gids[t], ref.ids):
            parity.assert_close(got[t], ref.out64, f"token {t} after a range error")


def test_prefill_input_beyond_fp16_range_reports_range_error():
    layer = synth.make_layer(synth.TINY, seed=0)
    x = synth.make_tokens(synth.TINY, seed=2, n_tokens=10)
    x[4, 17] = synth.bf16_bits(np.array([1.0e5], dtype=np.float32))[0]
    st, plan, scratch, dl = _status_after_prefill(layer, x)
    assert st == binding.SI_ERR_RANGE
    _prefill_again_is_correct(layer, plan, scratch, dl)


def test_prefill_h_beyond_fp16_range_reports_range_error():
    """Weights within fp16's range (d = 0.25, dmin = 0: |w| <= 236) whose
    SwiGLU output h = silu(g) * u reaches millions for N(0,1) tokens."""
    layer = synth.make_layer(synth.TINY, seed=0)
    big = synth.make_layer(synth.TINY, seed=0)
    for w in (big.w_gate, big.w_up):
        w[..., 0:2] = np.array([0.25], dtype="<f2").view(np.uint8)
        w[..., 2:4] = 0
    x = synth.make_tokens(synth.TINY, seed=2, n_tokens=10)
    st, plan, scratch, _ = _status_after_prefill(big, x)
    assert st == binding.SI_ERR_RANGE
    _prefill_again_is_correct(layer, plan, scratch, device.to_device(layer))


def test_prefill_weight_beyond_fp16_range_reports_range_error():
    """A block scale d = 65504 (the largest finite fp16): d*sc*q overflows fp16."""
    layer = synth.make_layer(synth.TINY, seed=0)
    bad = synth.make_layer(synth.TINY, seed=0)
    bad.w_down[:, 100, 0, 0:2] = np.array([65504.0], dtype="<f2").view(np.uint8)  # in every expert
    bad.w_down[:, 100, 0, 4:16] = 0xFF  # every 6-bit scale 63
    x = synth.make_tokens(synth.TINY, seed=2, n_tokens=10)
    st, plan, scratch, _ = _status_after_prefill(bad, x)
    assert st == binding.SI_ERR_RANGE
    _prefill_again_is_correct(layer, plan, scratch, device.to_device(layer))
