"""GB300-native Q4_K mixture-of-experts FFN: bs=1 decode (router, top-k,
dequant-on-read expert GEMVs, SwiGLU, weighted combine), small-batch
deduplicated decode and grouped prefill, behind the C ABI in
include/si_moe.h (libsimoe.so, built for sm_103a).

Modules:
  binding  -- ctypes binding with the C entry points' names
  device   -- moving synthetic layers/tokens into torch device memory
  synth    -- seeded synthetic inputs (shared with the CPU oracle)
  build    -- nvcc build of libsimoe.so

Importing the package loads nothing; the first binding call loads
libsimoe.so and raises if it has not been built.
"""
__all__ = ["binding", "device", "synth", "build"]
