"""The C-ABI library builds, loads and exports every symbol its header
declares (no GPU needed: no compute call is made)."""
import ctypes
import subprocess

import pytest

from quantized_moe_expert_gemv_gb300 import binding, build


@pytest.fixture(scope="module")
def lib():
    path = build.build()
    return binding.load_library(path)


def test_header_declares_the_boundary():
    names = binding.declared_symbols()
    for required in ("si_moe_plan", "si_moe_plan_destroy", "si_moe_scratch_bytes", "si_moe_scratch_init",
                     "si_moe_forward_decode", "si_moe_forward_prefill", "si_moe_read_status",
                     "si_status_string", "si_debug_q4k_dequant", "si_debug_topk"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", binding.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in binding.declared_symbols():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_status_strings(lib):
    for st in range(8):
        s = binding.si_status_string(st)
        assert isinstance(s, str) and s
    assert binding.si_status_string(binding.SI_ERR_MISALIGNED).startswith("device pointer")


def test_plan_rejects_bad_descriptors_before_touching_a_device(lib):
    D = binding.make_desc
    bad = [
        (D(300, 768, 128, 8), binding.SI_ERR_INVALID_ARG),        # hidden not a multiple of 256
        (D(2048, 700, 128, 8), binding.SI_ERR_INVALID_ARG),       # intermediate not a multiple of 256
        (D(2048, 768, 0, 1), binding.SI_ERR_INVALID_ARG),
        (D(2048, 768, 257, 8), binding.SI_ERR_INVALID_ARG),       # more experts than supported
        (D(2048, 768, 8, 9), binding.SI_ERR_INVALID_ARG),         # k > E
        (D(2048, 768, 128, 17), binding.SI_ERR_INVALID_ARG),      # k above the maximum
        (D(2048, 768, 128, 0), binding.SI_ERR_INVALID_ARG),
        (D(2048, 768, 128, 8, max_tokens=0), binding.SI_ERR_INVALID_ARG),
        (D(2048, 768, 128, 8, wtype=2), binding.SI_ERR_UNSUPPORTED),   # not Q4_K
        (D(2048, 768, 128, 8, flags=2), binding.SI_ERR_UNSUPPORTED),   # an unknown flag
        (D(2048, 768, 128, 8, wtype=binding.SI_WTYPE_NVFP4, flags=binding.SI_FLAG_ACT_INT8),
         binding.SI_ERR_UNSUPPORTED),                                  # int8 activations: Q4_K only
    ]
    for desc, want in bad:
        assert binding.si_moe_plan_status(desc) == want
    h = ctypes.c_void_p()
    assert lib.si_moe_plan(None, 0, ctypes.byref(h)) == binding.SI_ERR_INVALID_ARG
    assert lib.si_moe_plan(ctypes.byref(D(256, 256, 8, 2)), 0, None) == binding.SI_ERR_INVALID_ARG


def test_null_plan_arguments_are_rejected(lib):
    size = ctypes.c_size_t()
    assert lib.si_moe_scratch_bytes(None, 0, 1, ctypes.byref(size)) == binding.SI_ERR_INVALID_ARG
    assert lib.si_moe_read_status(None, None, None) == binding.SI_ERR_INVALID_ARG
    assert lib.si_moe_forward_decode(None, None, None, 1, None, None, None, 0, None) == \
        binding.SI_ERR_INVALID_ARG
    assert lib.si_moe_forward_prefill(None, None, None, 1, None, None, None, 0, None) == \
        binding.SI_ERR_INVALID_ARG
    assert lib.si_moe_forward_decode_host(None, None, None, 1, None, None, None, 0, None) == \
        binding.SI_ERR_INVALID_ARG
    assert lib.si_debug_q4k_dequant(None, 1, None, None, None) == binding.SI_ERR_INVALID_ARG
    assert lib.si_debug_q4k_dequant(16, 1, 17, None, None) == binding.SI_ERR_MISALIGNED
