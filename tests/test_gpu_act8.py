"""GPU checks of the int8-activation decode mode (SI_FLAG_ACT_INT8) through the
C ABI.  The mode is an approximation with its own tolerance, reported
separately from the default path:
  * against the oracle's emulation of the mode (oracle.moe_token_act8: the
    same int8 quantisation of x and h, exact integer dot products) the GPU
    output agrees to EMU_REL_L2 -- what remains is fp32 arithmetic and, rarely,
    an h value rounding to the neighbouring int8 code;
  * against the exact block (oracle.moe_token) the error of the mode itself
    is measured and held to ACT8_REL_L2 (a loose sanity bound; typical
    values are 1e-3 .. 1e-2).
Routing is unchanged (fp32 logits), so the ids follow the default rules."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from quantized_moe_expert_gemv_gb300 import binding, build, device, synth
from tests import parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

EMU_REL_L2 = 5e-4
EMU_MAX_REL = 3e-3
ACT8_REL_L2 = 0.15


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    binding.load_library()
    oracle.build()


def _plan(shape, flags=binding.SI_FLAG_ACT_INT8, max_tokens=1):
    return binding.si_moe_plan(device.desc_for(shape, max_tokens=max_tokens, flags=flags))


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


def _check_tokens(layer, x, outs, ids, w):
    s = layer.shape
    o_ids, o_w, z64, margin = oracle.route_tokens(layer.router_w, x, s.top_k, want_logits=True)
    checked, errs = 0, []
    for t in range(x.shape[0]):
        if not parity.routing_ok(ids[t], o_ids[t], z64[t], margin[t], s.top_k):
            continue
        parity.same_by_id(ids[t], w[t], o_ids[t], o_w[t], atol=2e-6)
        _, _, emu = oracle.moe_token_act8(layer, x[t])
        r = parity.rel_l2(outs[t], emu)
        m = float(np.abs(outs[t] - emu).max() / np.abs(emu).max())
        assert r <= EMU_REL_L2 and m <= EMU_MAX_REL, f"token {t}: vs emulation rel_l2={r:.3e} max_rel={m:.3e}"
        errs.append(parity.rel_l2(outs[t], oracle.moe_token(layer, x[t]).out64))
        checked += 1
    assert checked >= 1
    assert max(errs) <= ACT8_REL_L2, errs
    return errs


@pytest.mark.parametrize("shape,n_tok", [(synth.QWEN3_30B_A3B, 12), (synth.TINY, 8),
                                         (synth.MoeShape(1024, 768, 32, 8), 4), (synth.MoeShape(512, 512, 64, 6), 4)])
def test_act8_single_token_decode_matches_the_emulation(shape, n_tok):
    layer = synth.make_layer(shape, seed=shape.hidden + shape.n_experts)
    plan = _plan(shape)
    assert binding.si_debug_decode_fused(plan, 1) == 2  # the cluster expert kernel serves one token
    dl = device.to_device(layer)
    scratch = device.alloc_scratch(plan, binding.SI_MODE_DECODE, 1)
    x = synth.make_tokens(shape, seed=7, n_tokens=n_tok)
    res = [_decode(plan, dl, x[t:t + 1], shape, scratch) for t in range(n_tok)]
    _check_tokens(layer, x, np.concatenate([r[0] for r in res]), np.concatenate([r[1] for r in res]),
                  np.concatenate([r[2] for r in res]))


@pytest.mark.parametrize("n", [2, 4])
def test_act8_flag_leaves_batched_decode_unchanged(n):
    """Batched decode keeps its int16 activations under the flag: the same
    kernel and routing, outputs equal up to the order of the float reductions
    of the top-k combine (they vary from run to run)."""
    shape = synth.QWEN3_30B_A3B
    layer = synth.make_layer(shape, seed=3)
    dl = device.to_device(layer)
    x = synth.make_tokens(shape, seed=8, n_tokens=n)
    plan8, plan0 = _plan(shape), _plan(shape, flags=0)
    assert binding.si_debug_decode_fused(plan8, n) == binding.si_debug_decode_fused(plan0, n)
    a = _decode(plan8, dl, x, shape)
    b = _decode(plan0, dl, x, shape)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])   # routing: bit-exact
    for t in range(n):
        assert parity.rel_l2(a[0][t], b[0][t]) < 1e-6


def test_act8_flag_leaves_prefill_unchanged():
    shape = synth.MoeShape(512, 768, 16, 4)
    layer = synth.make_layer(shape, seed=9)
    dl = device.to_device(layer)
    T = 70
    x = device.tokens_to_device(synth.make_tokens(shape, seed=9, n_tokens=T))
    outs = []
    for flags in (binding.SI_FLAG_ACT_INT8, 0):
        plan = _plan(shape, flags=flags, max_tokens=T)
        scratch = device.alloc_scratch(plan, binding.SI_MODE_PREFILL, T)
        out = torch.empty((T, shape.hidden), dtype=torch.float32, device="cuda")
        binding.si_moe_forward_prefill(plan, dl.struct(), x, T, out, None, scratch)
        assert binding.si_moe_read_status(plan, scratch) == binding.SI_OK
        outs.append(out.cpu().numpy())
    assert np.array_equal(outs[0], outs[1])


def test_act8_with_a_prenormed_block_is_unsupported():
    shape = synth.TINY
    layer = synth.make_layer(shape, seed=0)
    dl = device.to_device(layer)
    plan = _plan(shape)
    scratch = device.alloc_scratch(plan, binding.SI_MODE_DECODE, 1)
    x = device.tokens_to_device(synth.make_tokens(shape, seed=0, n_tokens=1))
    out = torch.empty((1, shape.hidden), dtype=torch.float32, device="cuda")
    gamma = torch.ones(shape.hidden, dtype=torch.float32, device="cuda")
    normed = binding.layer_struct(dl.w_gate, dl.w_up, dl.w_down, dl.router_w, None, gamma, 1e-6)
    assert binding.si_moe_forward_decode(plan, normed, x, 1, out, None, scratch,
                                         raw_status=True) == binding.SI_ERR_UNSUPPORTED
