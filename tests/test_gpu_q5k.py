"""GPU parity of Q5_K experts (GGUF's 176-byte K-quant block) against the CPU
oracle, through the C ABI: the prefill operand conversion bit for bit,
single-token decode (cluster kernel), 2..4-token decode (generic kernels) and
the grouped prefill, under the default tolerance rules."""
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
    return device.desc_for(shape, max_tokens=max_tokens, wtype=binding.SI_WTYPE_Q5_K)


def _decode(plan, dl, x_bits, shape, scratch=None):
    n = x_bits.shape[0]
    scratch = scratch if scratch is not None else device.alloc_scratch(plan, binding.SI_MODE_DECODE, n)
    out = torch.full((n, shape.hidden), float("nan"), dtype=torch.float32, device="cuda")
    ids = torch.full((n, shape.top_k), -1, dtype=torch.int32, device="cuda")
    w = torch.empty((n, shape.top_k), dtype=torch.float32, device="cuda")
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
        parity.assert_close(out[t], oracle.moe_token(layer, x_bits[t]).out64, f"q5k token {t}")
        checked += 1
    assert checked >= 1
    assert np.isfinite(out).all()


def _special_q5k_blocks():
    g = synth.rng(71)
    b = synth.q5k_random_blocks(g, 64)
    b[0, 16:48] = 0xFF                       # every fifth bit set: codes 16..31
    b[1, 16:48] = 0x00                       # none set
    b[2, 16:48] = np.arange(32, dtype=np.uint8) * 8 + 1
    b[3, 0:2] = np.array([0xFF, 0x7B], dtype=np.uint8)  # largest finite fp16 d (range flag, finite fp32)
    b[4, 0:2] = np.array([0x01, 0x00], dtype=np.uint8)  # subnormal d
    b[5, 0:2] = np.array([0x00, 0xBC], dtype=np.uint8)  # negative d (-1)
    b[6, 2:4] = np.array([0x00, 0x00], dtype=np.uint8)  # dmin 0
    b[7, 4:16] = 0xFF                        # largest scales and mins
    return b


@pytest.mark.parametrize("with_gamma", [False, True])
def test_q5k_prefill_operand_conversion_bit_exact_against_oracle(with_gamma):
    blocks = np.concatenate([_special_q5k_blocks(), synth.q5k_random_blocks(synth.rng(72), 3000)])
    n = blocks.shape[0]
    ref = oracle.q5k_dequant(blocks).astype(np.float32)
    gamma = None
    if with_gamma:
        gamma = synth.rng(73).uniform(0.5, 1.5, n * 256).astype(np.float32)
        ref = (ref * gamma).astype(np.float32)
    out = torch.empty(n * 256, dtype=torch.int16, device="cuda")
    g_dev = None if gamma is None else torch.from_numpy(gamma).cuda()
    binding.si_debug_q5k_dequant_f16(torch.from_numpy(blocks).cuda(), n, g_dev, out)
    torch.cuda.synchronize()
    with np.errstate(over="ignore"):
        want = ref.astype(np.float16).view(np.uint16)
    got = out.cpu().numpy().view(np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (bad[:8], got[bad[:8]], want[bad[:8]])


def test_q5k_decode_qwen3_shape_single_tokens_take_the_cluster_kernel():
    shape = synth.QWEN3_30B_A3B
    layer = synth.make_layer_q5k(shape, seed=1)
    plan = binding.si_moe_plan(_desc(shape))
    assert binding.si_debug_decode_fused(plan, 1) == 2
    dl = device.to_device(layer)
    scratch = device.alloc_scratch(plan, binding.SI_MODE_DECODE, 1)
    x = synth.make_tokens(shape, seed=1, n_tokens=10)
    res = [_decode(plan, dl, x[t:t + 1], shape, scratch) for t in range(10)]
    _check(layer, x, np.concatenate([r[0] for r in res]), np.concatenate([r[1] for r in res]),
           np.concatenate([r[2] for r in res]))


@pytest.mark.parametrize("H,I,E,k", [(256, 256, 8, 2), (512, 256, 16, 4), (1024, 768, 32, 8)])
def test_q5k_decode_shapes(H, I, E, k):
    shape = synth.MoeShape(H, I, E, k)
    layer = synth.make_layer_q5k(shape, seed=H + I + E)
    plan = binding.si_moe_plan(_desc(shape))
    dl = device.to_device(layer)
    x = synth.make_tokens(shape, seed=4, n_tokens=3)
    res = [_decode(plan, dl, x[t:t + 1], shape) for t in range(3)]
    _check(layer, x, np.concatenate([r[0] for r in res]), np.concatenate([r[1] for r in res]),
           np.concatenate([r[2] for r in res]))


@pytest.mark.parametrize("n", [2, 3, 4])
def test_q5k_decode_small_batches(n):
    shape = synth.QWEN3_30B_A3B
    layer = synth.make_layer_q5k(shape, seed=2)
    plan = binding.si_moe_plan(_desc(shape))
    assert binding.si_debug_decode_fused(plan, n) == 3  # the cluster kernel over the distinct experts
    x = synth.make_tokens(shape, seed=20 + n, n_tokens=n)
    out, ids, w = _decode(plan, device.to_device(layer), x, shape)
    _check(layer, x, out, ids, w)


def test_q5k_decode_batched_identical_tokens():
    """Four copies of one token: every unit of the multi-token kernel (Q5_K blocks,
    its own cluster size) takes all four tokens."""
    shape = synth.QWEN3_30B_A3B
    layer = synth.make_layer_q5k(shape, seed=6)
    plan = binding.si_moe_plan(_desc(shape))
    assert binding.si_debug_decode_fused(plan, 4) == 3
    dl = device.to_device(layer)
    x1 = synth.make_tokens(shape, seed=6, n_tokens=1)
    x = np.repeat(x1, 4, axis=0)
    out, ids, w = _decode(plan, dl, x, shape)
    o1, i1, w1 = _decode(plan, dl, x1, shape)
    for t in range(4):
        assert np.array_equal(ids[t], i1[0])
        parity.assert_close(out[t], o1[0], "batched copy vs single")
    _check(layer, x, out, ids, w)


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


@pytest.mark.parametrize("H,I,E,k,T", [(256, 256, 8, 2, 41), (512, 768, 16, 4, 300)])
def test_q5k_prefill_ragged(H, I, E, k, T):
    shape = synth.MoeShape(H, I, E, k)
    layer = synth.make_layer_q5k(shape, seed=T)
    x = synth.make_tokens(shape, seed=T, n_tokens=T)
    out, ids, w = _prefill(layer, x)
    g = np.random.default_rng(T)
    _check(layer, x, out, ids, w, sorted(set(g.choice(T, size=min(T, 16), replace=False).tolist()) | {0, T - 1}))


def test_q5k_prefill_qwen3_workload_sampled():
    shape = synth.QWEN3_30B_A3B
    T = 4096
    layer = synth.make_layer_q5k(shape, seed=4)
    x = synth.make_tokens(shape, seed=4, n_tokens=T)
    out, ids, w = _prefill(layer, x)
    g = np.random.default_rng(9)
    _check(layer, x, out, ids, w, sorted(set(g.choice(T, size=16, replace=False).tolist()) | {0, T - 1}))


def test_q5k_with_a_prenormed_block_is_unsupported():
    shape = synth.TINY
    layer = synth.make_layer_q5k(shape, seed=0)
    dl = device.to_device(layer)
    plan = binding.si_moe_plan(_desc(shape))
    scratch = device.alloc_scratch(plan, binding.SI_MODE_DECODE, 1)
    x = device.tokens_to_device(synth.make_tokens(shape, seed=0, n_tokens=1))
    out = torch.empty((1, shape.hidden), dtype=torch.float32, device="cuda")
    gamma = torch.ones(shape.hidden, dtype=torch.float32, device="cuda")
    normed = binding.layer_struct(dl.w_gate, dl.w_up, dl.w_down, dl.router_w, None, gamma, 1e-6)
    assert binding.si_moe_forward_decode(plan, normed, x, 1, out, None, scratch,
                                         raw_status=True) == binding.SI_ERR_UNSUPPORTED
