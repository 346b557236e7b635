"""GPU parity of NVFP4 experts (E2M1 codes, E4M3 per-16 scales, fp32 tensor
scale per expert matrix) against the CPU oracle, through the C ABI: the
prefill operand conversion bit for bit, single-token decode (cluster kernel),
2..4-token decode (generic kernels) and the grouped prefill."""
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


def _desc(shape, max_tokens=1):
    return device.desc_for(shape, max_tokens=max_tokens, wtype=binding.SI_WTYPE_NVFP4)


def _decode(layer, x_bits, dl=None, plan=None, scratch=None):
    s = layer.shape
    n = x_bits.shape[0]
    dl = dl or device.to_device(layer)
    plan = plan or binding.si_moe_plan(_desc(s))
    scratch = scratch if scratch is not None else device.alloc_scratch(plan, binding.SI_MODE_DECODE, n)
    out = torch.full((n, s.hidden), float("nan"), dtype=torch.float32, device="cuda")
    ids = torch.full((n, s.top_k), -1, dtype=torch.int32, device="cuda")
    w = torch.empty((n, s.top_k), dtype=torch.float32, device="cuda")
    binding.si_moe_forward_decode(plan, dl.struct(), device.tokens_to_device(x_bits), n, out,
                                  binding.route_struct(topk_ids=ids, topk_w=w), scratch)
    assert binding.si_moe_read_status(plan, scratch) == binding.SI_OK
    return out.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy()


def _check(layer, x_bits, out, ids, w, sample=None):
    s = layer.shape
    o_ids, o_w, z64, margin = oracle.route_tokens(layer.router_w, x_bits, s.top_k, want_logits=True)
    checked = 0
    for t in (range(x_bits.shape[0]) if sample is None else sample):
        if not parity.routing_ok(ids[t], o_ids[t], z64[t], margin[t], s.top_k):
            continue
        parity.same_by_id(ids[t], w[t], o_ids[t], o_w[t], atol=2e-6)
        parity.assert_close(out[t], oracle.moe_token(layer, x_bits[t]).out64, f"nvfp4 token {t}")
        checked += 1
    assert checked >= 1
    assert np.isfinite(out).all()


# ------------------------------------------------ the prefill operand conversion
def test_nvfp4_prefill_operand_conversion_bit_exact_against_oracle():
    g = synth.rng(61)
    blocks = synth.nvfp4_random_blocks(g, 3000)
    # scale bytes across the E4M3 range: subnormals, the largest finite, negatives, zero
    blocks[0, 0:16] = [0x01, 0x02, 0x07, 0x08, 0x7E, 0x77, 0x00, 0x80, 0x81, 0xB8, 0xFE, 0x38, 0x3F, 0x40, 0x47, 0x5A]
    blocks[1, 16:] = np.arange(128, dtype=np.uint8)  # every code in both nibbles
    dev = torch.from_numpy(blocks).cuda()
    for gsc in (np.float32(1.0), np.float32(1.0 / 3.0), np.float32(0.0123), np.float32(-2.5)):
        ref = oracle.nvfp4_dequant(blocks, float(gsc))
        out = torch.empty(ref.size, dtype=torch.int16, device="cuda")
        binding.si_debug_nvfp4_dequant_f16(dev, blocks.shape[0], float(gsc), out)
        torch.cuda.synchronize()
        with np.errstate(over="ignore"):
            want = ref.astype(np.float16).view(np.uint16)
        assert np.array_equal(out.cpu().numpy().view(np.uint16), want), float(gsc)


# --------------------------------------------------------------------- decode
def test_nvfp4_decode_tiny_layer():
    layer = synth.make_layer_nvfp4(synth.TINY, seed=0)
    x = synth.make_tokens(synth.TINY, seed=0, n_tokens=8)
    out = np.empty((8, 256), dtype=np.float32)
    ids = np.empty((8, 2), dtype=np.int32)
    w = np.empty((8, 2), dtype=np.float32)
    dl = device.to_device(layer)
    plan = binding.si_moe_plan(_desc(synth.TINY))
    scratch = device.alloc_scratch(plan, binding.SI_MODE_DECODE, 1)
    for t in range(8):
        out[t:t + 1], ids[t:t + 1], w[t:t + 1] = _decode(layer, x[t:t + 1], dl, plan, scratch)
    _check(layer, x, out, ids, w)


def test_nvfp4_decode_qwen3_shape_single_tokens_take_the_cluster_kernel():
    shape = synth.QWEN3_30B_A3B
    layer = synth.make_layer_nvfp4(shape, seed=1)
    plan = binding.si_moe_plan(_desc(shape))
    assert binding.si_debug_decode_fused(plan, 1) == 2
    x = synth.make_tokens(shape, seed=1, n_tokens=12)
    dl = device.to_device(layer)
    scratch = device.alloc_scratch(plan, binding.SI_MODE_DECODE, 1)
    res = [_decode(layer, x[t:t + 1], dl, plan, scratch) for t in range(12)]
    out = np.concatenate([r[0] for r in res])
    ids = np.concatenate([r[1] for r in res])
    w = np.concatenate([r[2] for r in res])
    _check(layer, x, out, ids, w)


@pytest.mark.parametrize("n", [2, 3, 4])
def test_nvfp4_decode_small_batches(n):
    shape = synth.QWEN3_30B_A3B
    layer = synth.make_layer_nvfp4(shape, seed=2)
    plan = binding.si_moe_plan(_desc(shape))
    assert binding.si_debug_decode_fused(plan, n) == 3  # the cluster kernel over the distinct experts
    x = synth.make_tokens(shape, seed=10 + n, n_tokens=n)
    out, ids, w = _decode(layer, x, plan=plan)
    _check(layer, x, out, ids, w)


def test_nvfp4_decode_batched_identical_tokens():
    """Four copies of one token: every unit of the multi-token kernel takes all four
    tokens (NVFP4 tensor scales per unit, the down scale on each token's weight)."""
    shape = synth.QWEN3_30B_A3B
    layer = synth.make_layer_nvfp4(shape, seed=5)
    plan = binding.si_moe_plan(_desc(shape))
    assert binding.si_debug_decode_fused(plan, 4) == 3
    x1 = synth.make_tokens(shape, seed=5, n_tokens=1)
    x = np.repeat(x1, 4, axis=0)
    dl = device.to_device(layer)
    out, ids, w = _decode(layer, x, dl, plan)
    o1, i1, w1 = _decode(layer, x1, dl, plan)
    for t in range(4):
        assert np.array_equal(ids[t], i1[0])
        parity.assert_close(out[t], o1[0], "batched copy vs single")
    _check(layer, x, out, ids, w)


@pytest.mark.parametrize("H,I,E,k", [(512, 256, 16, 4), (1024, 768, 32, 8), (256, 512, 8, 1)])
def test_nvfp4_decode_shapes(H, I, E, k):
    shape = synth.MoeShape(H, I, E, k)
    layer = synth.make_layer_nvfp4(shape, seed=H + I + E + k)
    x = synth.make_tokens(shape, seed=3, n_tokens=3)
    for t in range(3):
        out, ids, w = _decode(layer, x[t:t + 1])
        _check(layer, x[t:t + 1], out, ids, w)


def test_nvfp4_argument_errors():
    shape = synth.TINY
    layer = synth.make_layer_nvfp4(shape, seed=0)
    dl = device.to_device(layer)
    x = device.tokens_to_device(synth.make_tokens(shape, seed=0, n_tokens=1))
    out = torch.empty((1, shape.hidden), dtype=torch.float32, device="cuda")
    plan = binding.si_moe_plan(_desc(shape))
    scratch = device.alloc_scratch(plan, binding.SI_MODE_DECODE, 1)
    no_scale = binding.layer_struct(dl.w_gate, dl.w_up, dl.w_down, dl.router_w)
    assert binding.si_moe_forward_decode(plan, no_scale, x, 1, out, None, scratch,
                                         raw_status=True) == binding.SI_ERR_INVALID_ARG
    gamma = torch.ones(shape.hidden, dtype=torch.float32, device="cuda")
    normed = binding.layer_struct(dl.w_gate, dl.w_up, dl.w_down, dl.router_w, None, gamma, 1e-6, dl.w_scale)
    assert binding.si_moe_forward_decode(plan, normed, x, 1, out, None, scratch,
                                         raw_status=True) == binding.SI_ERR_UNSUPPORTED
    q4_plan = binding.si_moe_plan(device.desc_for(shape))
    assert binding.si_moe_forward_decode(q4_plan, dl.struct(), x, 1, out, None, scratch,
                                         raw_status=True) == binding.SI_ERR_INVALID_ARG  # Q4_K with scales
    assert binding.si_moe_read_status(plan, scratch) == binding.SI_OK


# -------------------------------------------------------------------- prefill
def _prefill(layer, x_bits):
    s = layer.shape
    T = x_bits.shape[0]
    dl = device.to_device(layer)
    plan = binding.si_moe_plan(_desc(s, max_tokens=T))
    scratch = device.alloc_scratch(plan, binding.SI_MODE_PREFILL, T)
    out = torch.full((T, s.hidden), float("nan"), dtype=torch.float32, device="cuda")
    ids = torch.full((T, s.top_k), -1, dtype=torch.int32, device="cuda")
    w = torch.empty((T, s.top_k), dtype=torch.float32, device="cuda")
    binding.si_moe_forward_prefill(plan, dl.struct(), device.tokens_to_device(x_bits), T, out,
                                   binding.route_struct(topk_ids=ids, topk_w=w), scratch)
    assert binding.si_moe_read_status(plan, scratch) == binding.SI_OK
    return out.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("H,I,E,k,T", [(256, 256, 8, 2, 37), (512, 768, 16, 4, 300)])
def test_nvfp4_prefill_ragged(H, I, E, k, T):
    shape = synth.MoeShape(H, I, E, k)
    layer = synth.make_layer_nvfp4(shape, seed=T)
    x = synth.make_tokens(shape, seed=T, n_tokens=T)
    out, ids, w = _prefill(layer, x)
    g = np.random.default_rng(T)
    sample = sorted(set(g.choice(T, size=min(T, 16), replace=False).tolist()) | {0, T - 1})
    _check(layer, x, out, ids, w, sample)


def test_nvfp4_prefill_qwen3_workload_sampled():
    shape = synth.QWEN3_30B_A3B
    T = 4096
    layer = synth.make_layer_nvfp4(shape, seed=4)
    x = synth.make_tokens(shape, seed=4, n_tokens=T)
    out, ids, w = _prefill(layer, x)
    g = np.random.default_rng(9)
    _check(layer, x, out, ids, w, sorted(set(g.choice(T, size=16, replace=False).tolist()) | {0, T - 1}))
