"""Test-side helpers that build Q4_K super-blocks from chosen fields.

The packer below writes the 6-bit scales and mins into the 12 scale bytes
the way the Q4_K format lays them out (GGUF): for sub-blocks j < 4 the six
bits sit in the low bits of bytes j (scale) and j + 4 (min); for j >= 4 the
low four bits sit in byte j + 4 (scale in its low nibble, min in its high
nibble) and the top two bits sit in the top two bits of byte j - 4 (scale)
and byte j (min).  It is an encoder, the inverse direction of the oracle's
decoder, used to build closed-form blocks.
"""
from __future__ import annotations

import numpy as np


def pack_scales(sc: list[int], m: list[int]) -> np.ndarray:
    assert len(sc) == 8 and len(m) == 8
    assert all(0 <= v < 64 for v in sc + m)
    s = np.zeros(12, dtype=np.uint8)
    for j in range(4):
        s[j] = sc[j] & 63
        s[j + 4] = m[j] & 63
    for j in range(4, 8):
        s[j + 4] = (sc[j] & 15) | ((m[j] & 15) << 4)
        s[j - 4] |= (sc[j] >> 4) << 6
        s[j] |= (m[j] >> 4) << 6
    return s


def f16_bytes(value: float) -> np.ndarray:
    return np.array([value], dtype="<f2").view(np.uint8)


def make_block(d: float, dmin: float, sc: list[int], m: list[int], codes: np.ndarray) -> np.ndarray:
    """codes: [8, 32] 4-bit values q[j][l] for sub-block j, weight l."""
    codes = np.asarray(codes, dtype=np.uint8)
    assert codes.shape == (8, 32) and codes.max() < 16
    blk = np.zeros(144, dtype=np.uint8)
    blk[0:2] = f16_bytes(d)
    blk[2:4] = f16_bytes(dmin)
    blk[4:16] = pack_scales(sc, m)
    for i in range(4):
        blk[16 + 32 * i: 16 + 32 * i + 32] = codes[2 * i] | (codes[2 * i + 1] << 4)
    return blk


def dequant_test_blocks() -> np.ndarray:
    """The block set of the bit-exact dequantization tests, uint8 [n, 144]:
    the tiny layer's gate and down blocks, 5000 random blocks, one closed-form
    block per sub-block (a single nonzero scale, one nonzero min elsewhere,
    scales that set the two high bits) and blocks with special fp16 values of
    d and dmin (subnormals, zero, the largest finite value, negative)."""
    from quantized_moe_expert_gemv_gb300 import synth
    g = synth.rng(100)
    tiny = synth.make_layer(synth.TINY, seed=0)
    parts = [tiny.w_gate.reshape(-1, 144), tiny.w_down.reshape(-1, 144), synth.q4k_random_blocks(g, 5000)]
    for j in range(8):
        sc = [0] * 8
        sc[j] = 63 - j
        m = [0] * 8
        m[(j + 3) % 8] = 40 + j
        parts.append(make_block(0.0017, 0.0009, sc, m, np.full((8, 32), j + 3))[None])
    spec = synth.q4k_random_blocks(g, 6)
    for i, (dh, mh) in enumerate([(0x0001, 0x03ff), (0x0000, 0x0400), (0x7bff, 0x0000),
                                  (0x3c00, 0x3c00), (0x8001, 0x0002), (0x1234, 0xb800)]):
        spec[i, 0:2] = np.array([dh & 255, dh >> 8], dtype=np.uint8)
        spec[i, 2:4] = np.array([mh & 255, mh >> 8], dtype=np.uint8)
    parts.append(spec)
    return np.ascontiguousarray(np.concatenate(parts, axis=0))
