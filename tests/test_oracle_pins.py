"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each test ties one oracle function to the Q4_K definition through hand
arithmetic, a closed form, an invariant, a library routine or a brute-force
dense restatement, so that a dropped term, a wrong sign or index, or a
transposed operand anywhere in the oracle fails at least one test.
"""
from __future__ import annotations

import json
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.special

import oracle
from quantized_moe_expert_gemv_gb300 import synth
from tests.q4k_fixtures import make_block, pack_scales

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- fp16 / bf16
def test_half_to_double_matches_numpy_for_every_bit_pattern(oracle_lib):
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got) & (got > 0), np.isinf(ref) & (ref > 0))


def test_bf16_generator_matches_torch_rounding():
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(7)
    a = np.concatenate([g.standard_normal(100000).astype(np.float32),
                        np.array([0.0, -0.0, 1.0, 3.0e38, 1.0e-39], dtype=np.float32)])
    ours = synth.bf16_bits(a)
    ref = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert oracle.bf16_to_double(int(ours[0])) == float(torch.from_numpy(a[:1]).to(torch.bfloat16).float())


# ------------------------------------------------------------ scale/min unpack
def _bits(v: int) -> str:
    return format(v, "08b")


def _expected_sc_m(s: np.ndarray, j: int) -> tuple[int, int]:
    """The 6-bit fields read as bit strings (most significant bit first)."""
    if j < 4:
        return int(_bits(s[j])[2:], 2), int(_bits(s[j + 4])[2:], 2)
    sc = _bits(s[j - 4])[:2] + _bits(s[j + 4])[4:]
    m = _bits(s[j])[:2] + _bits(s[j + 4])[:4]
    return int(sc, 2), int(m, 2)


def test_scale_min_exhaustive_over_every_byte_read(oracle_lib):
    g = np.random.default_rng(1)
    for j in range(8):
        s = g.integers(0, 256, 12, dtype=np.uint8)
        if j < 4:
            for a in range(256):
                s[j] = a
                s[j + 4] = 255 - a
                assert oracle.q4k_scale_min(s, j) == _expected_sc_m(s, j)
        else:
            for a in range(256):
                for b in range(256):
                    s[j + 4] = a
                    s[j - 4] = b
                    s[j] = (a * 7 + b * 13) & 255
                    assert oracle.q4k_scale_min(s, j) == _expected_sc_m(s, j)


def test_scale_min_is_a_bijection_on_the_12_scale_bytes(oracle_lib):
    """16 six-bit fields fill exactly 96 bits: decoding then re-packing any 12
    bytes returns them unchanged, and packing then decoding returns the fields."""
    g = np.random.default_rng(2)
    for _ in range(2000):
        s = g.integers(0, 256, 12, dtype=np.uint8)
        sc, m = zip(*[oracle.q4k_scale_min(s, j) for j in range(8)])
        assert np.array_equal(pack_scales(list(sc), list(m)), s)
        sc2 = list(g.integers(0, 64, 8))
        m2 = list(g.integers(0, 64, 8))
        packed = pack_scales(sc2, m2)
        assert [oracle.q4k_scale_min(packed, j) for j in range(8)] == list(zip(sc2, m2))


# --------------------------------------------------------- hand-derived blocks
def _hand_block(spec) -> np.ndarray:
    blk = np.zeros(144, dtype=np.uint8)
    blk[0:2] = np.frombuffer(bytes.fromhex(spec["d_hex"])[::-1], dtype=np.uint8)
    blk[2:4] = np.frombuffer(bytes.fromhex(spec["dmin_hex"])[::-1], dtype=np.uint8)
    blk[4:16] = np.frombuffer(bytes.fromhex(spec["scales_hex"]), dtype=np.uint8)
    rule = spec["qs_rule"]
    if rule.startswith("qs[32i+l] = ((15 - l%16) << 4)"):
        for i in range(4):
            for l in range(32):
                blk[16 + 32 * i + l] = ((15 - l % 16) << 4) | (l % 16)
    elif rule.startswith("qs[0] = 0x01"):
        blk[16] = 0x01
    elif rule.startswith("all qs bytes 0xFF"):
        blk[16:] = 0xFF
    else:
        raise AssertionError(rule)
    return blk


def test_hand_derived_blocks(oracle_lib):
    with open(os.path.join(GOLDEN, "q4k_hand_blocks.json")) as f:
        fixture = json.load(f)
    n_checked = 0
    for spec in fixture["blocks"]:
        w = oracle.q4k_dequant(_hand_block(spec))
        for e in spec["expected"]:
            assert w[32 * e["j"] + e["l"]] == np.float32(e["w"]), (spec["name"], e)
            n_checked += 1
    assert n_checked >= 15


# --------------------------------------------------------- closed-form blocks
@pytest.mark.parametrize("j", range(8))
def test_single_nonzero_scale_closed_form(oracle_lib, j):
    d = 0.0013
    d16 = float(np.float16(d))
    for sc_val in (1, 17, 33, 48, 63):          # 17..63 set the high two bits for j >= 4
        for c in (1, 7, 15):
            sc = [0] * 8
            sc[j] = sc_val
            blk = make_block(d, 0.0, sc, [0] * 8, np.full((8, 32), c))
            w = oracle.q4k_dequant(blk).reshape(8, 32)
            expect = np.float32(d16 * sc_val * c)
            assert np.all(w[j] == expect)
            others = np.delete(w, j, axis=0)
            assert np.all(others == 0.0)


@pytest.mark.parametrize("j", range(8))
def test_min_only_closed_form(oracle_lib, j):
    dmin16 = float(np.float16(0.00071))
    for m_val in (1, 20, 47, 63):
        m = [0] * 8
        m[j] = m_val
        blk = make_block(0.002, 0.00071, [0] * 8, m, np.full((8, 32), 9))
        w = oracle.q4k_dequant(blk).reshape(8, 32)
        assert np.all(w[j] == np.float32(-dmin16 * m_val))
        assert np.all(np.delete(w, j, axis=0) == 0.0)


def test_nibble_order_and_position(oracle_lib):
    """Weight l of sub-block 2i is the low nibble of qs[32i+l]; of 2i+1 the high nibble."""
    codes = np.zeros((8, 32), dtype=np.uint8)
    for j in range(8):
        for l in range(32):
            codes[j, l] = (3 * j + 5 * l) % 16
    blk = make_block(1.0, 0.0, [1] * 8, [0] * 8, codes)
    w = oracle.q4k_dequant(blk).reshape(8, 32)
    assert np.array_equal(w, codes.astype(np.float32))
    # and directly from the bytes
    qs = blk[16:]
    for i in range(4):
        for l in range(32):
            assert w[2 * i, l] == qs[32 * i + l] & 15
            assert w[2 * i + 1, l] == qs[32 * i + l] >> 4


def test_dequant_is_the_exactly_rounded_value(oracle_lib):
    """Random blocks: each weight equals the exact rational d*sc*q - dmin*m
    rounded once to fp32."""
    g = synth.rng(11)
    blocks = synth.q4k_random_blocks(g, 40)
    w = oracle.q4k_dequant(blocks).reshape(40, 8, 32)
    for b in range(40):
        blk = blocks[b]
        d = Fraction(float(blk[0:2].view("<f2")[0]))
        dmin = Fraction(float(blk[2:4].view("<f2")[0]))
        s = blk[4:16]
        for j in range(8):
            sc, m = _expected_sc_m(s, j)
            for l in range(0, 32, 5):
                byte = int(blk[16 + 32 * (j // 2) + l])
                q = (byte & 15) if j % 2 == 0 else (byte >> 4)
                exact = d * sc * q - dmin * m
                assert w[b, j, l] == np.float32(float(exact))


# --------------------------------------------------------------------- routing
def test_router_logits_match_numpy(oracle_lib):
    g = np.random.default_rng(3)
    E, H = 16, 512
    W = g.normal(0, 0.02, (E, H)).astype(np.float32)
    xb = synth.bf16_bits(g.standard_normal(H).astype(np.float32))
    bias = g.normal(0, 0.5, E).astype(np.float32)
    xf = synth.bf16_to_f32(xb).astype(np.float64)
    z = oracle.router_logits(W, xb, bias)
    ref = W.astype(np.float64) @ xf + bias.astype(np.float64)
    np.testing.assert_allclose(z, ref, rtol=1e-13, atol=1e-15)
    z0 = oracle.router_logits(W, xb)
    np.testing.assert_allclose(z0, W.astype(np.float64) @ xf, rtol=1e-13, atol=1e-15)


def test_topk_matches_stable_sort_with_ties(oracle_lib):
    g = np.random.default_rng(4)
    for E, k in ((8, 2), (128, 8), (256, 8), (16, 16), (5, 1)):
        for _ in range(50):
            z = g.integers(-6, 6, E).astype(np.float32) * np.float32(0.25)   # many exact ties
            ids = oracle.topk(z, k)
            ref = np.lexsort((np.arange(E), -z))[:k]     # descending value, then lower index
            assert np.array_equal(ids, ref)


def test_renormalised_weights(oracle_lib):
    g = np.random.default_rng(5)
    for E, k in ((8, 2), (128, 8), (32, 32)):
        z = g.normal(0, 1, E)
        ids = oracle.topk(z.astype(np.float32), k)
        w = oracle.renorm_weights(z, ids)
        assert abs(w.sum() - 1.0) < 1e-12
        # renormalising the full softmax = softmax over the selected logits
        np.testing.assert_allclose(w, scipy.special.softmax(z[ids]), rtol=1e-12)
        if k == E:
            np.testing.assert_allclose(w, scipy.special.softmax(z)[ids], rtol=1e-12)
        assert np.all(np.diff(w) <= 0)                 # descending logits -> descending weights


def test_route_tokens_margin_and_consistency(oracle_lib):
    g = np.random.default_rng(6)
    E, H, k, T = 32, 256, 4, 20
    W = g.normal(0, 0.02, (E, H)).astype(np.float32)
    xb = synth.bf16_bits(g.standard_normal((T, H)).astype(np.float32))
    ids, w, z, margin = oracle.route_tokens(W, xb, k, want_logits=True)
    for t in range(T):
        zs = np.sort(z[t])[::-1]
        assert margin[t] == zs[k - 1] - zs[k]
        assert np.array_equal(ids[t], oracle.topk(z[t].astype(np.float32), k))
        np.testing.assert_allclose(w[t], scipy.special.softmax(z[t][ids[t]]), rtol=1e-12)
        assert len(set(ids[t].tolist())) == k and ids[t].min() >= 0 and ids[t].max() < E


# ---------------------------------------------------------------- expert FFN
def _const_matrix(rows, cols, d, sc_j, j, code):
    """Q4_K matrix whose every block has one nonzero sub-block j (scale sc_j, code)."""
    sc = [0] * 8
    sc[j] = sc_j
    blk = make_block(d, 0.0, sc, [0] * 8, np.full((8, 32), code))
    return np.tile(blk, (rows, cols // 256, 1)).reshape(rows, cols // 256, 144)


@pytest.mark.parametrize("sign_case", ["positive", "negative_gate"])
def test_expert_ffn_closed_form(oracle_lib, sign_case):
    """x = ones: g = (H/256)*32*d*sc*c, u = (H/256)*32*d_u, h = silu(g)*u,
    y_c = (I/256)*32*d_d*sc_d*h for every output c."""
    H, I = 512, 256
    d16 = float(np.float16(0.0011))
    du16 = float(np.float16(0.03125))
    dd16 = float(np.float16(0.0019))
    wg = _const_matrix(I, H, 0.0011, 33, 5, 7)
    if sign_case == "negative_gate":
        # dmin*m dominates: every gate weight is -dmin*m (sc = 0)
        blk = make_block(0.001, 0.0005, [0] * 8, [40] * 8, np.full((8, 32), 3))
        wg = np.tile(blk, (I, H // 256, 1)).reshape(I, H // 256, 144)
        w_gate_val = -float(np.float16(0.0005)) * 40
        g_val = H * w_gate_val
    else:
        g_val = (H // 256) * 32 * d16 * 33 * 7
    wu = _const_matrix(I, H, 0.03125, 1, 0, 1)
    wd = _const_matrix(H, I, 0.0019, 9, 3, 2)
    x = np.ones(H)
    h, y = oracle.expert_ffn(wg, wu, wd, x, H, I)
    u_val = (H // 256) * 32 * du16
    h_val = g_val * scipy.special.expit(g_val) * u_val
    y_val = (I // 256) * 32 * dd16 * 9 * 2 * h_val
    np.testing.assert_allclose(h, h_val, rtol=1e-13)
    np.testing.assert_allclose(y, y_val, rtol=1e-13)
    # silu identity: silu(g) - silu(-g) = g
    assert abs(g_val * scipy.special.expit(g_val) - (-g_val) * scipy.special.expit(-g_val) - g_val) < 1e-9


def _dense_reference(layer, xb):
    """Brute force: every expert's FFN densely with numpy, then mask to the
    top-k and weight by the renormalised softmax."""
    s = layer.shape
    E, H, I, k = s.n_experts, s.hidden, s.intermediate, s.top_k
    x = synth.bf16_to_f32(xb).astype(np.float64)
    z = layer.router_w.astype(np.float64) @ x
    if layer.router_bias is not None:
        z = z + layer.router_bias.astype(np.float64)
    order = np.lexsort((np.arange(E), -z.astype(np.float32)))
    sel = order[:k]
    p = scipy.special.softmax(z)
    wsel = p[sel] / p[sel].sum()
    out = np.zeros(H)
    for e in range(E):
        Wg = oracle.q4k_dequant(layer.w_gate[e]).reshape(I, H).astype(np.float64)
        Wu = oracle.q4k_dequant(layer.w_up[e]).reshape(I, H).astype(np.float64)
        Wd = oracle.q4k_dequant(layer.w_down[e]).reshape(H, I).astype(np.float64)
        g = Wg @ x
        hh = g * scipy.special.expit(g) * (Wu @ x)
        y = Wd @ hh
        mask = np.isin(e, sel)
        if mask:
            out += wsel[list(sel).index(e)] * y
    return sel, wsel, out


@pytest.mark.parametrize("shape", [synth.MoeShape(256, 256, 4, 2), synth.MoeShape(512, 256, 4, 4),
                                   synth.MoeShape(256, 512, 6, 3)])
def test_moe_token_matches_dense_brute_force(oracle_lib, shape):
    layer = synth.make_layer(shape, seed=21)
    xs = synth.make_tokens(shape, seed=21, n_tokens=3)
    for t in range(3):
        res = oracle.moe_token(layer, xs[t])
        sel, wsel, out = _dense_reference(layer, xs[t])
        assert np.array_equal(res.ids, sel)
        np.testing.assert_allclose(res.w, wsel, rtol=1e-12)
        np.testing.assert_allclose(res.out64, out, rtol=1e-10, atol=1e-12 * np.abs(out).max())
        assert np.array_equal(res.out32, res.out64.astype(np.float32))


def test_identical_experts_reduce_to_one_expert(oracle_lib):
    shape = synth.MoeShape(256, 256, 6, 3)
    layer = synth.make_layer(shape, seed=22)
    for name in ("w_gate", "w_up", "w_down"):
        arr = getattr(layer, name)
        arr[:] = arr[0]
    xs = synth.make_tokens(shape, seed=22, n_tokens=4)
    for t in range(4):
        res = oracle.moe_token(layer, xs[t])
        x = synth.bf16_to_f32(xs[t]).astype(np.float64)
        _, y = oracle.expert_ffn(layer.w_gate[0], layer.w_up[0], layer.w_down[0], x, 256, 256)
        np.testing.assert_allclose(res.out64, y, rtol=1e-12, atol=1e-12 * np.abs(y).max())


def test_router_bias_shifts_selection(oracle_lib):
    shape = synth.MoeShape(256, 256, 8, 2)
    layer = synth.make_layer(shape, seed=23, router_bias=np.array([0, 0, 0, 0, 0, 50.0, 0, 40.0]))
    xs = synth.make_tokens(shape, seed=23, n_tokens=5)
    for t in range(5):
        res = oracle.moe_token(layer, xs[t])
        assert list(res.ids) == [5, 7]


# ------------------------------------------------ pre-normed block + residual
def test_rmsnorm_closed_forms(oracle_lib):
    import math
    three_four = synth.bf16_bits(np.array([3.0, 4.0], dtype=np.float32))
    xn = oracle.rmsnorm(three_four, np.array([1.0, 2.0], dtype=np.float32), 0.0)
    # mean square 12.5: 3 / sqrt(12.5) = 3 sqrt(2) / 5, 2 * 4 / sqrt(12.5) = 8 sqrt(2) / 5
    np.testing.assert_allclose(xn, [3 * math.sqrt(2) / 5, 8 * math.sqrt(2) / 5], rtol=1e-15)
    c = synth.bf16_bits(np.full(64, -2.5, dtype=np.float32))
    gam = np.linspace(0.5, 1.5, 64).astype(np.float32)
    np.testing.assert_allclose(oracle.rmsnorm(c, gam, 0.0), -gam.astype(np.float64), rtol=1e-15)
    eps = 0.75
    np.testing.assert_allclose(oracle.rmsnorm(c, gam, eps), -2.5 * gam.astype(np.float64) / math.sqrt(6.25 + eps),
                               rtol=1e-15)
    # without eps the norm is invariant to scaling x by a power of two (exact in bf16 and fp64)
    xs = synth.make_tokens(synth.MoeShape(256, 256, 4, 2), seed=31, n_tokens=1)[0]
    x2 = synth.bf16_bits(2.0 * synth.bf16_to_f32(xs))
    assert np.array_equal(oracle.rmsnorm(xs, gam.repeat(4), 0.0), oracle.rmsnorm(x2, gam.repeat(4), 0.0))


def test_prenorm_block_with_zero_experts_returns_the_residual(oracle_lib):
    shape = synth.MoeShape(256, 256, 4, 2)
    layer = synth.make_layer(shape, seed=32)
    for name in ("w_gate", "w_up", "w_down"):
        getattr(layer, name)[:] = 0  # d = dmin = 0: every weight is 0
    xs = synth.make_tokens(shape, seed=32, n_tokens=3)
    gam = synth.make_norm_weight(shape, seed=32)
    for t in range(3):
        res = oracle.moe_token_prenorm(layer, xs[t], gam, 1e-6)
        assert np.array_equal(res.out32, synth.bf16_to_f32(xs[t]))


def test_prenorm_block_on_unit_rms_input_is_x_plus_the_plain_block(oracle_lib):
    """x of +-1 entries has mean square 1; with gain 1 and eps 0 the norm is the
    identity, so the block is x + (the plain MoE FFN of x)."""
    shape = synth.MoeShape(512, 256, 6, 3)
    layer = synth.make_layer(shape, seed=33)
    g = np.random.default_rng(33)
    for _ in range(3):
        x = synth.bf16_bits(g.choice([-1.0, 1.0], size=shape.hidden).astype(np.float32))
        res = oracle.moe_token_prenorm(layer, x, np.ones(shape.hidden, np.float32), 0.0)
        plain = oracle.moe_token(layer, x)
        assert np.array_equal(res.ids, plain.ids)
        np.testing.assert_allclose(res.w, plain.w, rtol=1e-13)
        np.testing.assert_allclose(res.out64, synth.bf16_to_f32(x) + plain.out64, rtol=1e-12,
                                   atol=1e-12 * np.abs(plain.out64).max())


def test_prenorm_routing_agrees_with_the_block(oracle_lib):
    shape = synth.MoeShape(256, 256, 12, 3)
    layer = synth.make_layer(shape, seed=35, router_bias=np.linspace(0.0, 0.2, 12))
    gam = synth.make_norm_weight(shape, seed=35)
    xs = synth.make_tokens(shape, seed=35, n_tokens=5)
    ids, w, z, margin = oracle.route_tokens_prenorm(layer.router_w, xs, 3, gam, 1e-6, bias=layer.router_bias)
    for t in range(5):
        res = oracle.moe_token_prenorm(layer, xs[t], gam, 1e-6)
        assert np.array_equal(ids[t], res.ids)
        assert np.array_equal(w[t], res.w) and np.array_equal(z[t], res.z)
        assert margin[t] == res.margin
    # x of +-1 with unit gain and no eps: the plain routing of x
    x = synth.bf16_bits(np.random.default_rng(35).choice([-1.0, 1.0], size=(4, 256)).astype(np.float32))
    a = oracle.route_tokens_prenorm(layer.router_w, x, 3, np.ones(256, np.float32), 0.0, bias=layer.router_bias)
    b = oracle.route_tokens(layer.router_w, x, 3, bias=layer.router_bias, want_logits=True)
    assert np.array_equal(a[0], b[0])
    np.testing.assert_allclose(a[2], b[2], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(a[3], b[3], rtol=1e-9, atol=1e-13)


def test_prenorm_block_is_scale_invariant_up_to_the_residual(oracle_lib):
    """eps = 0: block(2x) - 2x = block(x) - x (the norm removes the scale, the
    residual keeps it)."""
    shape = synth.MoeShape(256, 512, 8, 2)
    layer = synth.make_layer(shape, seed=34, router_bias=np.linspace(-0.1, 0.1, 8))
    gam = synth.make_norm_weight(shape, seed=34)
    xs = synth.make_tokens(shape, seed=34, n_tokens=3)
    for t in range(3):
        x2 = synth.bf16_bits(2.0 * synth.bf16_to_f32(xs[t]))
        a = oracle.moe_token_prenorm(layer, xs[t], gam, 0.0)
        b = oracle.moe_token_prenorm(layer, x2, gam, 0.0)
        assert np.array_equal(a.ids, b.ids)
        xa = synth.bf16_to_f32(xs[t]).astype(np.float64)
        np.testing.assert_allclose(b.out64 - 2 * xa, a.out64 - xa, rtol=1e-11,
                                   atol=1e-11 * np.abs(a.out64 - xa).max())


# --------------------------------------------------------- prefill bookkeeping
def test_counts_offsets_perm_match_numpy(oracle_lib):
    g = np.random.default_rng(8)
    for T, k, E in ((1, 1, 1), (7, 2, 8), (300, 8, 128), (64, 4, 5)):
        ids = np.stack([g.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
        counts, offsets, perm = oracle.counts_offsets_perm(ids, E)
        flat = ids.reshape(-1)
        assert np.array_equal(counts, np.bincount(flat, minlength=E))
        assert offsets[0] == 0 and np.array_equal(offsets[1:], np.cumsum(counts))
        assert np.array_equal(perm, np.argsort(flat, kind="stable"))
        assert np.array_equal(np.sort(perm), np.arange(T * k))


# ------------------------------------------------------ dedup workload recipe
def test_stored_dedup_beta_gives_sixty_percent_hot_mass(oracle_lib):
    wl = synth.WORKLOADS["dedup4"]
    shape, seed = wl["shape"], wl["seed"]
    beta = synth.load_dedup_beta()
    bias = synth.dedup_router_bias(seed, beta)
    rw = synth.make_router_w(shape, seed)
    xs = synth.make_tokens(shape, seed, wl["tokens_per_step"] * wl["n_steps"])
    ids, w, _, _ = oracle.route_tokens(rw, xs, shape.top_k, bias=bias)
    hot = np.isin(ids, synth.dedup_hot_set(seed))
    share = float((w * hot).sum() / w.sum())
    assert abs(share - 0.60) <= 0.005, share


# ------------------------------------------------------------------------ NVFP4
# The E2M1 element values as the format's value table lists them (codes 0-7,
# then the same magnitudes negated for codes 8-15).
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def _nvfp4_block(scales16, codes256) -> np.ndarray:
    """Pack 16 E4M3 scale bytes and 256 4-bit codes into this library's NVFP4 super-block."""
    codes = np.asarray(codes256, dtype=np.uint8)
    blk = np.zeros(144, dtype=np.uint8)
    blk[0:16] = np.asarray(scales16, dtype=np.uint8)
    blk[16:] = codes[0::2] | (codes[1::2] << 4)
    return blk


def test_e2m1_values_match_the_format_table(oracle_lib):
    got = [oracle.e2m1_to_double(c) for c in range(16)]
    assert got == E2M1_TABLE
    assert [np.signbit(v) for v in got] == [c >= 8 for c in range(16)]


def test_e4m3_matches_torch_for_every_byte(oracle_lib):
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = b.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(i) for i in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.signbit(got[fin]), np.signbit(ref[fin]))
    assert oracle.e4m3_to_double(0x7E) == 448.0 and oracle.e4m3_to_double(0x01) == 2.0 ** -9


def test_nvfp4_element_order_scale_blocks_and_tensor_scale(oracle_lib):
    """Weight i of a super-block is code i (low nibble of byte 16 + i/2 for even
    i) times the E4M3 scale of block i/16 times the tensor scale."""
    codes = np.arange(256) % 16
    scales = [0x38 + 8 * (j % 4) for j in range(16)]      # 1, 2, 4, 8, 1, 2, ...
    blk = _nvfp4_block(scales, codes)
    for g in (1.0, 0.5, 3.0):
        w = oracle.nvfp4_dequant(blk, g)
        want = np.array([E2M1_TABLE[codes[i]] * (2.0 ** ((i // 16) % 4)) * g for i in range(256)], dtype=np.float32)
        assert np.array_equal(w, want)
    # a single nonzero scale: only its 16 weights survive
    for j in (0, 7, 15):
        sc = [0] * 16
        sc[j] = 0x40  # 2.0
        w = oracle.nvfp4_dequant(_nvfp4_block(sc, np.full(256, 7)), 1.0)  # every code 6.0
        assert np.array_equal(np.nonzero(w)[0], np.arange(16 * j, 16 * j + 16))
        assert np.all(w[16 * j: 16 * j + 16] == 12.0)


def test_nvfp4_dequant_is_the_exactly_rounded_value(oracle_lib):
    """Random super-blocks and tensor scales: each weight equals the exact
    rational e2m1 * e4m3 * g rounded once to fp32."""
    g = synth.rng(31)
    blocks = synth.nvfp4_random_blocks(g, 12)
    blocks[0, 0:16] = [0x01, 0x07, 0x08, 0x7E, 0xFE, 0x30, 0x00, 0x81, 0x39, 0x3A, 0x3B, 0x3C, 0x3D, 0x3E, 0x3F, 0x40]
    for gs in (np.float32(1.0 / 3.0), np.float32(0.0123), np.float32(7.77)):
        w = oracle.nvfp4_dequant(blocks, float(gs)).reshape(12, 256)
        for b in range(12):
            for i in range(0, 256, 3):
                code = (blocks[b, 16 + i // 2] >> (4 * (i % 2))) & 15
                sb = int(blocks[b, i // 16])
                sign = -1 if sb & 0x80 else 1
                E, M = (sb >> 3) & 15, sb & 7
                scale = Fraction(M, 8) * Fraction(1, 64) if E == 0 else (1 + Fraction(M, 8)) * Fraction(2) ** (E - 7)
                exact = Fraction(E2M1_TABLE[code]) * sign * scale * Fraction(float(gs))
                assert w[b, i] == np.float32(float(exact)), (b, i)


def _dequant_any(layer, name, e):
    arr = getattr(layer, name)[e]
    if layer.wtype == synth.WTYPE_NVFP4:
        k = {"w_gate": 0, "w_up": 1, "w_down": 2}[name]
        return oracle.nvfp4_dequant(arr, float(layer.gscale[e, k]))
    return oracle.q4k_dequant(arr)


@pytest.mark.parametrize("shape", [synth.MoeShape(256, 256, 4, 2), synth.MoeShape(512, 256, 5, 3)])
def test_nvfp4_moe_token_matches_dense_brute_force(oracle_lib, shape):
    layer = synth.make_layer_nvfp4(shape, seed=33)
    H, I, E, k = shape.hidden, shape.intermediate, shape.n_experts, shape.top_k
    xs = synth.make_tokens(shape, seed=33, n_tokens=3)
    for t in range(3):
        res = oracle.moe_token(layer, xs[t])
        x = synth.bf16_to_f32(xs[t]).astype(np.float64)
        z = layer.router_w.astype(np.float64) @ x
        sel = np.argsort(-z.astype(np.float32), kind="stable")[:k]
        p = scipy.special.softmax(z)
        wsel = p[sel] / p[sel].sum()
        out = np.zeros(H)
        for e in range(E):  # every expert, masked afterwards
            Wg = _dequant_any(layer, "w_gate", e).reshape(I, H).astype(np.float64)
            Wu = _dequant_any(layer, "w_up", e).reshape(I, H).astype(np.float64)
            Wd = _dequant_any(layer, "w_down", e).reshape(H, I).astype(np.float64)
            gg = Wg @ x
            y = Wd @ (gg * scipy.special.expit(gg) * (Wu @ x))
            if e in sel:
                out += wsel[list(sel).index(e)] * y
        assert np.array_equal(res.ids, sel)
        np.testing.assert_allclose(res.out64, out, rtol=1e-10, atol=1e-12 * np.abs(out).max())


def test_nvfp4_identical_experts_reduce_to_one_expert(oracle_lib):
    shape = synth.MoeShape(256, 256, 6, 3)
    layer = synth.make_layer_nvfp4(shape, seed=34)
    for name in ("w_gate", "w_up", "w_down"):
        arr = getattr(layer, name)
        arr[:] = arr[0]
    layer.gscale[:] = layer.gscale[0]
    xs = synth.make_tokens(shape, seed=34, n_tokens=3)
    for t in range(3):
        res = oracle.moe_token(layer, xs[t])
        x = synth.bf16_to_f32(xs[t]).astype(np.float64)
        _, y = oracle.expert_ffn(layer.w_gate[0], layer.w_up[0], layer.w_down[0], x, 256, 256,
                                 wtype=oracle.WTYPE_NVFP4, gscales=layer.gscale[0])
        np.testing.assert_allclose(res.out64, y, rtol=1e-12, atol=1e-12 * np.abs(y).max())


# ----------------------------------------------------------------- int8-activation mode
def _rne(fr: Fraction) -> int:
    """Round a rational to the nearest integer, ties to even."""
    fl = fr.numerator // fr.denominator
    rem = fr - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        return fl + 1
    return fl


def test_act8_quant_rules(oracle_lib):
    g = np.random.default_rng(81)
    v = (g.standard_normal(32 * 40) * np.exp(g.uniform(-6, 6, 32 * 40))).astype(np.float32)
    v[32 * 3:32 * 4] = 0.0                       # an all-zero block
    v[32 * 5:32 * 6] = np.float32(-1e-3)         # a constant negative block
    v[32 * 7:32 * 8] = np.array([127.0] + [2.5, 3.5, -4.5, 0.5, -0.5, 1.5, -1.5] + [0.0] * 24, dtype=np.float32)
    q, d, s = oracle.act8_quant(v)
    for b in range(40):
        blk = v[32 * b:32 * b + 32]
        mx = np.float32(np.abs(blk).max())
        assert d[b] == np.float32(mx * np.float32(1.0 / 127.0))
        assert s[b] == sum(Fraction(float(t)) for t in blk)  # the exact sum (32 fp32 values fit in fp64 here)
        if mx == 0:
            assert not q[32 * b:32 * b + 32].any()
            continue
        inv = np.float32(127.0) / mx                 # fp32 division, correctly rounded
        want = [_rne(Fraction(float(t)) * Fraction(float(inv))) for t in blk]
        assert list(q[32 * b:32 * b + 32]) == want
        assert abs(int(q[32 * b + int(np.argmax(np.abs(blk)))])) == 127
        # reconstruction error within half a step (plus the rounding of inv)
        err = np.abs(blk.astype(np.float64) - float(d[b]) * q[32 * b:32 * b + 32])
        assert err.max() <= 0.5 * float(d[b]) * (1 + 1e-6) + 127 * float(d[b]) * 2e-7
    # ties go to the even integer (inv == 1 exactly in block 7)
    assert list(q[32 * 7:32 * 7 + 8]) == [127, 2, 4, -4, 0, 0, 2, -2]
    assert list(q[32 * 5:32 * 5 + 32]) == [-127] * 32


def _subblock_dm_dsc(blocks: np.ndarray):
    """(dsc, dm) of every 32-weight sub-block of Q4_K blocks [n][144], as fp32 products."""
    n = blocks.shape[0]
    dsc = np.empty((n, 8), dtype=np.float32)
    dm = np.empty((n, 8), dtype=np.float32)
    for i in range(n):
        dd = np.float32(oracle.half_to_double(int(blocks[i, 0]) | (int(blocks[i, 1]) << 8)))
        dmin = np.float32(oracle.half_to_double(int(blocks[i, 2]) | (int(blocks[i, 3]) << 8)))
        for j in range(8):
            sc, m = oracle.q4k_scale_min(blocks[i, 4:16], j)
            dsc[i, j] = dd * np.float32(sc)
            dm[i, j] = dmin * np.float32(m)
    return dsc, dm


def _act8_dot_dense(W, dm_rows, qv, dv, sv):
    """Rows of W (exact weights) against the quantised activation: the scale term
    on d*q and the min term on the exact block sums, written as the dense product
    with the quantised activation plus the min-term correction."""
    xhat = np.repeat(dv.astype(np.float64), 32) * qv.astype(np.float64)
    corr = dm_rows.astype(np.float64) @ (np.add.reduceat(xhat, np.arange(0, xhat.size, 32)) - sv)
    return W @ xhat + corr


def _q4k_w64(blocks: np.ndarray, rows: int):
    """Weights of Q4_K blocks [n][144] as fp64 dsc*c - dm (no rounding to fp32),
    the codes c read from the nibbles: qs[32i + l] = weight l of sub-blocks 2i
    (low nibble) and 2i+1 (high nibble)."""
    dsc, dm = _subblock_dm_dsc(blocks)
    qs = blocks[:, 16:].reshape(-1, 4, 32)
    codes = np.stack([qs & 15, qs >> 4], axis=2).reshape(-1, 8, 32).astype(np.float64)
    w = dsc.astype(np.float64)[:, :, None] * codes - dm.astype(np.float64)[:, :, None]
    return w.reshape(rows, -1), dm.reshape(rows, -1)


@pytest.mark.parametrize("H,I", [(256, 256), (512, 768)])
def test_act8_expert_ffn_matches_dense_rewrite(oracle_lib, H, I):
    shape = synth.MoeShape(H, I, 2, 1)
    layer = synth.make_layer(shape, seed=H + I)
    x = synth.make_tokens(shape, seed=5, n_tokens=1)[0]
    x64 = np.array([oracle.bf16_to_double(int(b)) for b in x])
    h, y = oracle.expert_ffn_act8(layer.w_gate[1], layer.w_up[1], layer.w_down[1], x64, H, I)
    # the same steps from pinned pieces: dense fp64 weights (before their fp32
    # rounding, which the mode does not take), the quantiser, per-sub-block dm
    Wg, dmg = _q4k_w64(np.asarray(layer.w_gate[1]).reshape(-1, 144), I)
    Wu, dmu = _q4k_w64(np.asarray(layer.w_up[1]).reshape(-1, 144), I)
    Wd, dmd = _q4k_w64(np.asarray(layer.w_down[1]).reshape(-1, 144), H)
    # those fp64 weights round to the oracle's fp32 ones
    assert np.array_equal(Wg.astype(np.float32).ravel(), oracle.q4k_dequant(layer.w_gate[1]))
    qx, dx, sx = oracle.act8_quant(x64.astype(np.float32))
    g = _act8_dot_dense(Wg, dmg, qx, dx, sx)
    u = _act8_dot_dense(Wu, dmu, qx, dx, sx)
    hh = g * scipy.special.expit(g) * u
    np.testing.assert_allclose(h, hh, rtol=1e-9, atol=1e-12 * np.abs(hh).max())
    qh, dh, shh = oracle.act8_quant(h.astype(np.float32))
    yy = _act8_dot_dense(Wd, dmd, qh, dh, shh)
    np.testing.assert_allclose(y, yy, rtol=1e-9, atol=1e-12 * np.abs(yy).max())


def test_act8_mode_error_against_the_exact_block(oracle_lib):
    """The approximation itself: same routing, output within about 1e-2 rel-L2 on
    these tokens (a token whose h has a large outlier in some 32-column block
    can reach several 1e-2 on larger layers; the mode is reported separately)."""
    shape = synth.MoeShape(512, 256, 8, 2)
    layer = synth.make_layer(shape, seed=33)
    xs = synth.make_tokens(shape, seed=33, n_tokens=4)
    errs = []
    for t in range(4):
        ids, w, out = oracle.moe_token_act8(layer, xs[t])
        ref = oracle.moe_token(layer, xs[t])
        assert np.array_equal(ids, ref.ids)
        np.testing.assert_allclose(w, ref.w, rtol=1e-12)
        errs.append(np.linalg.norm(out - ref.out64) / np.linalg.norm(ref.out64))
    assert 1e-4 < max(errs) < 3e-2


# ----------------------------------------------------------------- Q5_K
def _q5k_from_q4k(q4: np.ndarray, qh: np.ndarray) -> np.ndarray:
    """The Q5_K blocks with the Q4_K blocks' d, dmin, scales and qs and the given qh bytes."""
    n = q4.shape[0]
    out = np.zeros((n, 176), dtype=np.uint8)
    out[:, 0:16] = q4[:, 0:16]
    out[:, 16:48] = qh
    out[:, 48:176] = q4[:, 16:144]
    return out


def test_q5k_with_no_high_bits_is_q4k(oracle_lib):
    g = synth.rng(91)
    q4 = synth.q4k_random_blocks(g, 200)
    q5 = _q5k_from_q4k(q4, np.zeros((200, 32), dtype=np.uint8))
    assert np.array_equal(oracle.q5k_dequant(q5), oracle.q4k_dequant(q4))


def test_q5k_each_high_bit_adds_sixteen_steps_to_one_weight(oracle_lib):
    g = synth.rng(92)
    q4 = synth.q4k_random_blocks(g, 3)
    base_qh = np.zeros((3, 32), dtype=np.uint8)
    base = oracle.q5k_dequant(_q5k_from_q4k(q4, base_qh)).reshape(3, 256)
    for blk in range(3):
        dd = Fraction(oracle.half_to_double(int(q4[blk, 0]) | (int(q4[blk, 1]) << 8)))
        dmin = Fraction(oracle.half_to_double(int(q4[blk, 2]) | (int(q4[blk, 3]) << 8)))
        for j in range(8):
            sc, m = oracle.q4k_scale_min(q4[blk, 4:16], j)
            for l in (0, 5, 31):
                qh = base_qh.copy()
                qh[blk, l] = 1 << j
                got = oracle.q5k_dequant(_q5k_from_q4k(q4, qh)).reshape(3, 256)
                diff = np.nonzero(got != base)
                # only weight l of sub-block j of this block moved ...
                assert list(zip(*diff)) in ([(blk, 32 * j + l)], []), (blk, j, l, diff)
                # ... to the exactly rounded value of its code plus 16
                qs_byte = int(q4[blk, 16 + 32 * (j // 2) + l])
                code = (qs_byte >> 4 if j % 2 else qs_byte & 15) + 16
                want = float(np.float32(float(dd * sc * code - dmin * m)))
                assert got[blk, 32 * j + l] == want


@pytest.mark.parametrize("shape", [synth.MoeShape(256, 256, 4, 2), synth.MoeShape(512, 256, 6, 3)])
def test_q5k_moe_token_matches_dense_brute_force(oracle_lib, shape):
    layer = synth.make_layer_q5k(shape, seed=23)
    xs = synth.make_tokens(shape, seed=23, n_tokens=2)
    H, I = shape.hidden, shape.intermediate
    for t in range(2):
        res = oracle.moe_token(layer, xs[t])
        x = synth.bf16_to_f32(xs[t]).astype(np.float64)
        z = layer.router_w.astype(np.float64) @ x
        sel = oracle.topk(z.astype(np.float32), shape.top_k)
        p = np.exp(z[sel] - z[sel].max())
        wsel = p / p.sum()
        out = np.zeros(H)
        for e, w in zip(sel, wsel):
            Wg = oracle.q5k_dequant(layer.w_gate[e]).reshape(I, H).astype(np.float64)
            Wu = oracle.q5k_dequant(layer.w_up[e]).reshape(I, H).astype(np.float64)
            Wd = oracle.q5k_dequant(layer.w_down[e]).reshape(H, I).astype(np.float64)
            gg = Wg @ x
            out += w * (Wd @ (gg * scipy.special.expit(gg) * (Wu @ x)))
        assert np.array_equal(res.ids, sel)
        np.testing.assert_allclose(res.out64, out, rtol=1e-10, atol=1e-12 * np.abs(out).max())
