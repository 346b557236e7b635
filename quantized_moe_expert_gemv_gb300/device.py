"""Device residency for layers and tokens (torch owns the memory).

Weights stay in their quantized form in HBM (GGUF Q4_K blocks, or NVFP4
super-blocks), exactly the bytes the generator holds; nothing is
dequantized ahead of time.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

from . import binding
from .synth import MoeLayer, MoeShape


@dataclass
class DeviceLayer:
    shape: MoeShape
    w_gate: torch.Tensor      # uint8 [E, I, H/256, 144]
    w_up: torch.Tensor
    w_down: torch.Tensor      # uint8 [E, H, I/256, 144]
    router_w: torch.Tensor    # float32 [E, H]
    router_bias: Optional[torch.Tensor] = None
    norm_weight: Optional[torch.Tensor] = None   # float32 [H]: pre-normed block with residual
    norm_eps: float = 0.0
    w_scale: Optional[torch.Tensor] = None       # float32 [E, 3]: NVFP4 tensor scales

    def struct(self) -> binding.si_moe_layer:
        return binding.layer_struct(self.w_gate, self.w_up, self.w_down, self.router_w,
                                    self.router_bias, self.norm_weight, self.norm_eps, self.w_scale)

    @property
    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.w_gate, self.w_up, self.w_down,
                                                            self.router_w))


def to_device(layer: MoeLayer, device="cuda") -> DeviceLayer:
    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)
    bias = None if layer.router_bias is None else up(layer.router_bias)
    norm = None if layer.norm_weight is None else up(layer.norm_weight)
    wsc = None if getattr(layer, "gscale", None) is None else up(layer.gscale)
    return DeviceLayer(layer.shape, up(layer.w_gate), up(layer.w_up), up(layer.w_down),
                       up(layer.router_w), bias, norm, float(layer.norm_eps) if norm is not None else 0.0, wsc)


def tokens_to_device(x_bits: np.ndarray, device="cuda") -> torch.Tensor:
    """bf16 bit patterns (uint16 numpy) -> torch.bfloat16 device tensor."""
    t = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def desc_for(shape: MoeShape, max_tokens: int = 1, wtype: int = binding.SI_WTYPE_Q4_K,
             flags: int = 0) -> binding.si_moe_desc:
    return binding.make_desc(shape.hidden, shape.intermediate, shape.n_experts, shape.top_k, max_tokens, wtype,
                             flags)


def alloc_scratch(plan: binding.Plan, mode: int, n_tokens: int, device="cuda",
                  stream=None) -> torch.Tensor:
    nbytes = binding.si_moe_scratch_bytes(plan, mode, n_tokens)
    t = torch.empty(nbytes, dtype=torch.uint8, device=device)
    binding.si_moe_scratch_init(plan, t, stream)
    return t
