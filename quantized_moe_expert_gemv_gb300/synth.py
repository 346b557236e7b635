"""Seeded synthetic inputs for a Q4_K-resident mixture-of-experts FFN layer.

This module only draws random bytes and numbers. It holds none of the
method's arithmetic (no dequantization, routing, FFN or combine), so both
the CUDA path (tests, bench) and the CPU oracle (tests) may take their
inputs from it.

Value recipe (the sparkinfer pages name Q4_K_M experts, the Qwen3-30B-A3B
shape and greedy bs=1 decode, but print no weights; the recipe is the
plainest synthetic stand-in with the shapes of those workloads):
  * Q4_K super-block, 144 bytes per 256 weights, in GGUF byte order
    {fp16 d, fp16 dmin, u8 scales[12], u8 qs[128]}:
      d    ~ U[1e-4, 2e-3] rounded to fp16 (round-to-nearest-even),
      dmin ~ U[0, 1e-3]    rounded to fp16,
      scales[12], qs[128]: uniform random bytes.
  * router weights fp32 ~ N(0, 0.02); activations x ~ N(0, 1) rounded to
    bf16 (round-to-nearest-even), carried as uint16 bit patterns.

Weight tensors are expert-major and blocked along each matrix's input
(column) dimension, GGUF's own row layout:
  gate, up : [E][I rows][H/256 blocks][144 B]
  down     : [E][H rows][I/256 blocks][144 B]

Every draw comes from numpy's PCG64 seeded through SeedSequence with an
explicit key, which gives the same bytes on x86-64 and aarch64.
"""
from __future__ import annotations

import json
import os
from dataclasses import dataclass

import numpy as np

Q4K_BLOCK_BYTES = 144
Q4K_BLOCK_WEIGHTS = 256

_DIR = os.path.dirname(os.path.abspath(__file__))


@dataclass(frozen=True)
class MoeShape:
    hidden: int          # H: model dimension (input of gate/up, output of down)
    intermediate: int    # I: expert FFN width
    n_experts: int       # E
    top_k: int           # k

    @property
    def blocks_per_gate_row(self) -> int:
        return self.hidden // Q4K_BLOCK_WEIGHTS

    @property
    def blocks_per_down_row(self) -> int:
        return self.intermediate // Q4K_BLOCK_WEIGHTS

    @property
    def expert_bytes(self) -> int:
        """Q4_K bytes of one expert's gate + up + down matrices."""
        return 3 * self.hidden * self.intermediate // Q4K_BLOCK_WEIGHTS * Q4K_BLOCK_BYTES


# Tiny layer: hidden 256, 8 experts, top-2, intermediate 256, seed 0.
TINY = MoeShape(hidden=256, intermediate=256, n_experts=8, top_k=2)
# Qwen3-30B-A3B MoE layer: hidden 2048, 128 experts, top-8, intermediate 768.
QWEN3_30B_A3B = MoeShape(hidden=2048, intermediate=768, n_experts=128, top_k=8)


def rng(*key: int | str) -> np.random.Generator:
    """A PCG64 generator keyed by a tuple of ints/strings."""
    ints = []
    for k in key:
        if isinstance(k, str):
            ints.extend(k.encode())
        else:
            ints.append(int(k))
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(ints)))


def q4k_random_blocks(g: np.random.Generator, n_blocks: int) -> np.ndarray:
    """n_blocks random Q4_K super-blocks, uint8 [n_blocks, 144]."""
    raw = np.frombuffer(g.bytes(n_blocks * Q4K_BLOCK_BYTES), dtype=np.uint8)
    raw = raw.reshape(n_blocks, Q4K_BLOCK_BYTES).copy()
    d = g.uniform(1e-4, 2e-3, n_blocks).astype(np.float16)
    dmin = g.uniform(0.0, 1e-3, n_blocks).astype(np.float16)
    raw[:, 0:2] = d.astype("<f2").view(np.uint8).reshape(n_blocks, 2)
    raw[:, 2:4] = dmin.astype("<f2").view(np.uint8).reshape(n_blocks, 2)
    return raw


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest-even); return the uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


WTYPE_Q4_K = 12      # GGUF's type id of Q4_K
WTYPE_Q5_K = 13      # GGUF's type id of Q5_K (layout below)
WTYPE_NVFP4 = 100    # NVFP4 super-blocks (layout below)
Q5K_BLOCK_BYTES = 176


@dataclass
class MoeLayer:
    shape: MoeShape
    w_gate: np.ndarray        # uint8 [E, I, H/256, 144]
    w_up: np.ndarray          # uint8 [E, I, H/256, 144]
    w_down: np.ndarray        # uint8 [E, H, I/256, 144]
    router_w: np.ndarray      # float32 [E, H]
    router_bias: np.ndarray | None = None   # float32 [E] or None
    norm_weight: np.ndarray | None = None   # float32 [H] RMSNorm gain (pre-normed block) or None
    norm_eps: float = 1e-6
    wtype: int = WTYPE_Q4_K
    gscale: np.ndarray | None = None        # float32 [E, 3] NVFP4 tensor scales of gate, up, down


def make_router_w(shape: MoeShape, seed: int, layer: int = 0) -> np.ndarray:
    """Router weights fp32 N(0, 0.02), [E, H]."""
    g = rng(seed, layer, "router")
    return g.normal(0.0, 0.02, size=(shape.n_experts, shape.hidden)).astype(np.float32)


def make_layer(shape: MoeShape, seed: int, layer: int = 0,
               router_bias: np.ndarray | None = None) -> MoeLayer:
    E, H, I = shape.n_experts, shape.hidden, shape.intermediate
    nbh, nbi = shape.blocks_per_gate_row, shape.blocks_per_down_row
    wg = q4k_random_blocks(rng(seed, layer, "gate"), E * I * nbh).reshape(E, I, nbh, Q4K_BLOCK_BYTES)
    wu = q4k_random_blocks(rng(seed, layer, "up"), E * I * nbh).reshape(E, I, nbh, Q4K_BLOCK_BYTES)
    wd = q4k_random_blocks(rng(seed, layer, "down"), E * H * nbi).reshape(E, H, nbi, Q4K_BLOCK_BYTES)
    rw = make_router_w(shape, seed, layer)
    bias = None if router_bias is None else np.asarray(router_bias, dtype=np.float32).copy()
    return MoeLayer(shape, wg, wu, wd, rw, bias)


# ---------------------------------------------------------------------------
# NVFP4 experts: 4-bit E2M1 codes, one FP8 E4M3 scale per 16 weights and one
# fp32 scale per expert matrix, stored in super-blocks of 256 weights with the
# same size as a Q4_K block (144 bytes): bytes 0-15 the 16 E4M3 scales of
# weights 16j .. 16j+15, bytes 16-143 the codes (byte 16 + l holds weight 2l
# in its low nibble and weight 2l+1 in its high nibble).  Synthetic recipe:
# codes uniform random nibbles; block scales E4M3 with exponent field 7..9
# and a random mantissa (values in [1, 8)); tensor scales 2^-6 * U[0.5, 1.5]
# rounded to fp32, so weights have magnitudes like the Q4_K recipe's.
# ---------------------------------------------------------------------------
def nvfp4_random_blocks(g: np.random.Generator, n_blocks: int) -> np.ndarray:
    """n_blocks random NVFP4 super-blocks, uint8 [n_blocks, 144]."""
    raw = np.frombuffer(g.bytes(n_blocks * Q4K_BLOCK_BYTES), dtype=np.uint8)
    raw = raw.reshape(n_blocks, Q4K_BLOCK_BYTES).copy()
    exp = g.integers(7, 10, size=(n_blocks, 16), dtype=np.uint8)
    man = g.integers(0, 8, size=(n_blocks, 16), dtype=np.uint8)
    raw[:, 0:16] = (exp << 3) | man
    return raw


def make_layer_nvfp4(shape: MoeShape, seed: int, layer: int = 0,
                     router_bias: np.ndarray | None = None) -> MoeLayer:
    E, H, I = shape.n_experts, shape.hidden, shape.intermediate
    nbh, nbi = shape.blocks_per_gate_row, shape.blocks_per_down_row
    wg = nvfp4_random_blocks(rng(seed, layer, "nvfp4-gate"), E * I * nbh).reshape(E, I, nbh, Q4K_BLOCK_BYTES)
    wu = nvfp4_random_blocks(rng(seed, layer, "nvfp4-up"), E * I * nbh).reshape(E, I, nbh, Q4K_BLOCK_BYTES)
    wd = nvfp4_random_blocks(rng(seed, layer, "nvfp4-down"), E * H * nbi).reshape(E, H, nbi, Q4K_BLOCK_BYTES)
    gsc = (rng(seed, layer, "nvfp4-tensor-scale").uniform(0.5, 1.5, size=(E, 3)) / 64.0).astype(np.float32)
    rw = make_router_w(shape, seed, layer)
    bias = None if router_bias is None else np.asarray(router_bias, dtype=np.float32).copy()
    return MoeLayer(shape, wg, wu, wd, rw, bias, wtype=WTYPE_NVFP4, gscale=gsc)


def make_norm_weight(shape: MoeShape, seed: int, layer: int = 0) -> np.ndarray:
    """RMSNorm gain of a pre-normed block: fp32 U[0.5, 1.5], [H]."""
    g = rng(seed, layer, "norm")
    return g.uniform(0.5, 1.5, size=shape.hidden).astype(np.float32)


def make_tokens(shape: MoeShape, seed: int, n_tokens: int, stream: int | str = "x") -> np.ndarray:
    """bf16 activations N(0,1) as uint16 bits, [n_tokens, H]."""
    g = rng(seed, "tokens", stream)
    return bf16_bits(g.standard_normal((n_tokens, shape.hidden), dtype=np.float32))


# ---------------------------------------------------------------------------
# Biased routing for the small-batch dedup workload: a hot set of 32 of the
# 128 experts receives a constant logit offset beta.  The hot set is the first
# 32 entries of a seeded permutation; beta itself is a stored number, found
# once with the CPU oracle so that the hot set carries 60% of the
# renormalised top-k routing mass on the workload's 512 x 4 tokens (the
# script that wrote it lives under tests/golden/).
# ---------------------------------------------------------------------------
DEDUP_BIAS_FILE = os.path.join(os.path.dirname(_DIR), "tests", "golden", "dedup_bias.json")


def dedup_hot_set(seed: int, n_experts: int = 128, n_hot: int = 32) -> np.ndarray:
    return np.sort(rng(seed, "hot-set").permutation(n_experts)[:n_hot]).astype(np.int32)


def dedup_router_bias(seed: int, beta: float, n_experts: int = 128, n_hot: int = 32) -> np.ndarray:
    b = np.zeros(n_experts, dtype=np.float32)
    b[dedup_hot_set(seed, n_experts, n_hot)] = np.float32(beta)
    return b


def load_dedup_beta() -> float:
    with open(DEDUP_BIAS_FILE) as f:
        return float(json.load(f)["beta"])


# Workload descriptions (sizes and seeds); "seed" follows the workload's index.
WORKLOADS = {
    "tiny": dict(shape=TINY, seed=0, n_tokens=1),
    "layer": dict(shape=QWEN3_30B_A3B, seed=1, n_tokens=1024),
    "stack48": dict(shape=QWEN3_30B_A3B, seed=2, n_layers=48, n_steps=256),
    "dedup4": dict(shape=QWEN3_30B_A3B, seed=3, tokens_per_step=4, n_steps=512),
    "prefill": dict(shape=QWEN3_30B_A3B, seed=4, n_tokens=4096),
}


# ---------------------------------------------------------------------------
# Device-side drawing for the 48-layer stack (16 GB of Q4_K bytes): the same
# distributions as q4k_random_blocks, drawn by torch's CUDA generator so the
# stack is resident in seconds.  The oracle never reads these layers; parity
# of the per-layer kernels is established on numpy-drawn layers of the same
# shape.
# ---------------------------------------------------------------------------
def _torch_seed(*key) -> int:
    return int(rng(*key).integers(0, 2**62))


def q4k_random_blocks_torch(n_blocks: int, seed_key: tuple, device="cuda"):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(_torch_seed(*seed_key))
    raw = torch.randint(0, 256, (n_blocks, Q4K_BLOCK_BYTES), dtype=torch.uint8, device=device,
                        generator=g)
    d = (torch.rand(n_blocks, generator=g, device=device, dtype=torch.float32) * (2e-3 - 1e-4)
         + 1e-4).to(torch.float16)
    dmin = (torch.rand(n_blocks, generator=g, device=device, dtype=torch.float32) * 1e-3).to(torch.float16)
    raw[:, 0:2] = d.view(torch.uint8).view(n_blocks, 2)
    raw[:, 2:4] = dmin.view(torch.uint8).view(n_blocks, 2)
    return raw


def make_layer_torch(shape: MoeShape, seed: int, layer: int, device="cuda"):
    """(w_gate, w_up, w_down, router_w) as device tensors for one layer."""
    import torch
    E, H, I = shape.n_experts, shape.hidden, shape.intermediate
    nbh, nbi = shape.blocks_per_gate_row, shape.blocks_per_down_row
    wg = q4k_random_blocks_torch(E * I * nbh, (seed, layer, "gate-dev"), device).view(E, I, nbh, 144)
    wu = q4k_random_blocks_torch(E * I * nbh, (seed, layer, "up-dev"), device).view(E, I, nbh, 144)
    wd = q4k_random_blocks_torch(E * H * nbi, (seed, layer, "down-dev"), device).view(E, H, nbi, 144)
    g = torch.Generator(device=device)
    g.manual_seed(_torch_seed(seed, layer, "router-dev"))
    rw = torch.randn((E, H), generator=g, device=device, dtype=torch.float32) * 0.02
    return wg, wu, wd, rw


def make_tokens_torch(n: int, hidden: int, seed_key: tuple, device="cuda"):
    """bf16 N(0,1) activations [n, hidden] drawn on the device."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(_torch_seed(*seed_key))
    return torch.randn((n, hidden), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


# ---------------------------------------------------------------------------
# Q5_K experts (GGUF's Q5_K block, 176 bytes per 256 weights: d, dmin, the
# Q4_K scale/min bytes, qh[32] -- bit j of qh[l] is the value-16 bit of weight
# l of sub-block j -- and qs[128] arranged as Q4_K's).  Synthetic recipe: like
# q4k_random_blocks with uniform random qh and qs bytes and d ~ U[5e-5, 1e-3]
# (half the Q4_K range: the codes reach 31), dmin ~ U[0, 1e-3].
# ---------------------------------------------------------------------------
def q5k_random_blocks(g: np.random.Generator, n_blocks: int) -> np.ndarray:
    """n_blocks random Q5_K super-blocks, uint8 [n_blocks, 176]."""
    raw = np.frombuffer(g.bytes(n_blocks * Q5K_BLOCK_BYTES), dtype=np.uint8)
    raw = raw.reshape(n_blocks, Q5K_BLOCK_BYTES).copy()
    d = g.uniform(5e-5, 1e-3, n_blocks).astype(np.float16)
    dmin = g.uniform(0.0, 1e-3, n_blocks).astype(np.float16)
    raw[:, 0:2] = d.astype("<f2").view(np.uint8).reshape(n_blocks, 2)
    raw[:, 2:4] = dmin.astype("<f2").view(np.uint8).reshape(n_blocks, 2)
    return raw


def make_layer_q5k(shape: MoeShape, seed: int, layer: int = 0,
                   router_bias: np.ndarray | None = None) -> MoeLayer:
    E, H, I = shape.n_experts, shape.hidden, shape.intermediate
    nbh, nbi = shape.blocks_per_gate_row, shape.blocks_per_down_row
    wg = q5k_random_blocks(rng(seed, layer, "q5k-gate"), E * I * nbh).reshape(E, I, nbh, Q5K_BLOCK_BYTES)
    wu = q5k_random_blocks(rng(seed, layer, "q5k-up"), E * I * nbh).reshape(E, I, nbh, Q5K_BLOCK_BYTES)
    wd = q5k_random_blocks(rng(seed, layer, "q5k-down"), E * H * nbi).reshape(E, H, nbi, Q5K_BLOCK_BYTES)
    rw = make_router_w(shape, seed, layer)
    bias = None if router_bias is None else np.asarray(router_bias, dtype=np.float32).copy()
    return MoeLayer(shape, wg, wu, wd, rw, bias, wtype=WTYPE_Q5_K)
