"""Thin ctypes binding of libsimoe (include/si_moe.h).

The functions below carry the C entry points' names and only marshal
arguments: tensors become device pointers, torch streams become
cudaStream_t, and a non-OK status raises SiError.  Every step of the MoE
path runs in the library's CUDA kernels; there is no fallback.  If the
library has not been built, loading it raises immediately.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
LIB_PATH = os.path.join(PKG_DIR, "_build", "libsimoe.so")
HEADER_PATH = os.path.join(ROOT, "include", "si_moe.h")

SI_OK = 0
SI_ERR_INVALID_ARG = 1
SI_ERR_UNSUPPORTED = 2
SI_ERR_MISALIGNED = 3
SI_ERR_SCRATCH_TOO_SMALL = 4
SI_ERR_CUDA = 5
SI_ERR_TIMEOUT = 6
SI_ERR_DEVICE = 7
SI_ERR_RANGE = 8
SI_WTYPE_Q4_K = 12
SI_WTYPE_NVFP4 = 100
SI_WTYPE_Q5_K = 13
SI_FLAG_ACT_INT8 = 1
SI_MODE_DECODE = 0
SI_MODE_PREFILL = 1
SI_MODE_DECODE_HOST = 2
SI_MAX_EXPERTS = 256
SI_MAX_TOPK = 16
SI_MAX_DECODE_TOKENS = 4
SI_STATIC_SCRATCH_BYTES = 1 << 20


class SiError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {si_status_string(status)} (status {status})")


class si_moe_desc(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("intermediate", ctypes.c_int32),
                ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("max_tokens", ctypes.c_int32), ("wtype", ctypes.c_int32),
                ("flags", ctypes.c_uint32)]


class si_moe_layer(ctypes.Structure):
    _fields_ = [("w_gate", ctypes.c_void_p), ("w_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p),
                ("router_w", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
                ("norm_weight", ctypes.c_void_p), ("norm_eps", ctypes.c_float), ("w_scale", ctypes.c_void_p)]


class si_moe_route_out(ctypes.Structure):
    _fields_ = [("topk_ids", ctypes.c_void_p), ("topk_w", ctypes.c_void_p),
                ("expert_counts", ctypes.c_void_p), ("expert_offsets", ctypes.c_void_p),
                ("perm", ctypes.c_void_p), ("logits", ctypes.c_void_p)]


_lib = None


def library_path() -> str:
    return LIB_PATH


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libsimoe; raise if it is missing (build it first)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libsimoe is not built ({p} missing): run "
                           "`python -m quantized_moe_expert_gemv_gb300.build` first")
    lib = ctypes.CDLL(p)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.si_status_string.restype = ctypes.c_char_p
    lib.si_status_string.argtypes = [ctypes.c_int]
    lib.si_moe_plan.restype = ctypes.c_int
    lib.si_moe_plan.argtypes = [ctypes.POINTER(si_moe_desc), ctypes.c_int, ctypes.POINTER(vp)]
    lib.si_moe_plan_destroy.restype = None
    lib.si_moe_plan_destroy.argtypes = [vp]
    lib.si_moe_scratch_bytes.restype = ctypes.c_int
    lib.si_moe_scratch_bytes.argtypes = [vp, ctypes.c_int, i32, ctypes.POINTER(sz)]
    lib.si_moe_scratch_init.restype = ctypes.c_int
    lib.si_moe_scratch_init.argtypes = [vp, vp, sz, vp]
    for name in ("si_moe_forward_decode", "si_moe_forward_prefill", "si_moe_forward_decode_host"):
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        f.argtypes = [vp, ctypes.POINTER(si_moe_layer), vp, i32, vp, ctypes.POINTER(si_moe_route_out),
                      vp, sz, vp]
    lib.si_debug_decode_events.restype = ctypes.c_int
    lib.si_debug_decode_events.argtypes = [vp, ctypes.POINTER(si_moe_layer), vp, i32, vp,
                                           ctypes.POINTER(si_moe_route_out), vp, sz,
                                           ctypes.POINTER(vp), vp]
    lib.si_debug_prefill_events.argtypes = [vp, ctypes.POINTER(si_moe_layer), vp, i32, vp,
                                            ctypes.POINTER(si_moe_route_out), vp, sz,
                                            ctypes.POINTER(vp), vp]
    lib.si_debug_prefill_events.restype = ctypes.c_int
    lib.si_moe_forward_decode_noalloc.restype = ctypes.c_int
    lib.si_moe_forward_decode_noalloc.argtypes = [vp, ctypes.POINTER(si_moe_layer), vp, i32, vp,
                                                  ctypes.POINTER(si_moe_route_out), vp]
    lib.si_debug_plan_info.restype = ctypes.c_int
    lib.si_debug_plan_info.argtypes = [vp, ctypes.POINTER(i32), i32]
    lib.si_debug_decode_fused.restype = ctypes.c_int
    lib.si_debug_decode_fused.argtypes = [vp, i32]
    lib.si_moe_read_status.restype = ctypes.c_int
    lib.si_moe_read_status.argtypes = [vp, vp, vp]
    lib.si_debug_q4k_dequant.restype = ctypes.c_int
    lib.si_debug_q4k_dequant.argtypes = [vp, i64, vp, vp, vp]
    lib.si_debug_q4k_dequant_f16.restype = ctypes.c_int
    lib.si_debug_q4k_dequant_f16.argtypes = [vp, i64, vp, vp, vp]
    lib.si_debug_nvfp4_dequant_f16.restype = ctypes.c_int
    lib.si_debug_nvfp4_dequant_f16.argtypes = [vp, i64, ctypes.c_float, vp, vp]
    lib.si_debug_q5k_dequant_f16.restype = ctypes.c_int
    lib.si_debug_q5k_dequant_f16.argtypes = [vp, i64, vp, vp, vp]
    lib.si_moe_read_status_noalloc.restype = ctypes.c_int
    lib.si_moe_read_status_noalloc.argtypes = [vp]
    lib.si_debug_topk.restype = ctypes.c_int
    lib.si_debug_topk.argtypes = [vp, i32, ctypes.POINTER(si_moe_desc),
                                  ctypes.POINTER(si_moe_route_out), vp]
    if path is None:
        _lib = lib
    return lib


def declared_symbols() -> list[str]:
    """Names of the functions include/si_moe.h declares."""
    with open(HEADER_PATH) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:si_status|void|int|const char \*)\s*\*?\s*(si_\w+)\s*\(",
                                 text, flags=re.M)))


# ------------------------------------------------------------ marshalling
def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "__array_interface__"):  # a numpy array in host memory
        return t.__array_interface__["data"][0]
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != SI_OK:
        raise SiError(status, where)


def si_status_string(status: int) -> str:
    return load_library().si_status_string(int(status)).decode()


def make_desc(hidden, intermediate, n_experts, top_k, max_tokens=1, wtype=SI_WTYPE_Q4_K, flags=0):
    return si_moe_desc(hidden, intermediate, n_experts, top_k, max_tokens, wtype, flags)


class Plan:
    """Owns an si_moe_plan_t (host memory only)."""

    def __init__(self, handle: int, desc: si_moe_desc):
        self.handle = handle
        self.desc = desc

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.si_moe_plan_destroy(self.handle)
            self.handle = None


def si_moe_plan(desc: si_moe_desc, cuda_device: int = 0) -> Plan:
    h = ctypes.c_void_p()
    _check(load_library().si_moe_plan(ctypes.byref(desc), cuda_device, ctypes.byref(h)), "si_moe_plan")
    return Plan(h.value, desc)


def si_moe_plan_status(desc: si_moe_desc, cuda_device: int = 0) -> int:
    """si_moe_plan's status without raising (frees a plan it made)."""
    lib = load_library()
    h = ctypes.c_void_p()
    st = lib.si_moe_plan(ctypes.byref(desc), cuda_device, ctypes.byref(h))
    if st == SI_OK:
        lib.si_moe_plan_destroy(h)
    return st


def si_moe_scratch_bytes(plan: Plan, mode: int, n_tokens: int) -> int:
    out = ctypes.c_size_t()
    _check(load_library().si_moe_scratch_bytes(plan.handle, mode, n_tokens, ctypes.byref(out)),
           "si_moe_scratch_bytes")
    return out.value


def si_moe_scratch_init(plan: Plan, scratch, stream=None):
    _check(load_library().si_moe_scratch_init(plan.handle, _ptr(scratch), scratch.numel() *
                                              scratch.element_size(), _stream(stream)),
           "si_moe_scratch_init")


def layer_struct(w_gate, w_up, w_down, router_w, router_bias=None, norm_weight=None,
                 norm_eps: float = 0.0, w_scale=None) -> si_moe_layer:
    return si_moe_layer(_ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(router_w), _ptr(router_bias),
                        _ptr(norm_weight), float(norm_eps), _ptr(w_scale))


def route_struct(topk_ids=None, topk_w=None, expert_counts=None, expert_offsets=None, perm=None,
                 logits=None) -> si_moe_route_out:
    return si_moe_route_out(_ptr(topk_ids), _ptr(topk_w), _ptr(expert_counts), _ptr(expert_offsets),
                            _ptr(perm), _ptr(logits))


def _forward(fn_name, plan, layer, x, n_tokens, out, route_out, scratch, stream, raw_status):
    lib = load_library()
    ro = ctypes.byref(route_out) if route_out is not None else None
    nbytes = scratch.numel() * scratch.element_size()
    st = getattr(lib, fn_name)(plan.handle, ctypes.byref(layer), _ptr(x), int(n_tokens), _ptr(out), ro,
                               _ptr(scratch), nbytes, _stream(stream))
    if raw_status:
        return st
    _check(st, fn_name)
    return st


def si_moe_forward_decode(plan, layer: si_moe_layer, x, n_tokens, out, route_out=None, scratch=None,
                          stream=None, raw_status=False):
    return _forward("si_moe_forward_decode", plan, layer, x, n_tokens, out, route_out, scratch, stream,
                    raw_status)


def si_moe_forward_prefill(plan, layer: si_moe_layer, x, n_tokens, out, route_out=None, scratch=None,
                           stream=None, raw_status=False):
    return _forward("si_moe_forward_prefill", plan, layer, x, n_tokens, out, route_out, scratch, stream,
                    raw_status)


def si_moe_forward_decode_host(plan, layer: si_moe_layer, x_host, n_tokens, out_host, route_out=None,
                               scratch=None, stream=None, raw_status=False):
    """Decode with x and out in host memory (numpy arrays or CPU tensors);
    returns once out_host holds the result.  scratch:
    si_moe_scratch_bytes(plan, SI_MODE_DECODE_HOST, n)."""
    return _forward("si_moe_forward_decode_host", plan, layer, x_host, n_tokens, out_host, route_out, scratch,
                    stream, raw_status)


def si_moe_forward_decode_noalloc(plan, layer: si_moe_layer, x, n_tokens, out, route_out=None,
                                  stream=None, raw_status=False):
    """Decode with the library's built-in device scratch (no caller buffer,
    no allocation); see include/si_moe.h for its limits."""
    ro = ctypes.byref(route_out) if route_out is not None else None
    st = load_library().si_moe_forward_decode_noalloc(plan.handle, ctypes.byref(layer), _ptr(x),
                                                      int(n_tokens), _ptr(out), ro, _stream(stream))
    if not raw_status:
        _check(st, "si_moe_forward_decode_noalloc")
    return st


def si_debug_decode_events(plan, layer: si_moe_layer, x, n_tokens, out, route_out=None, scratch=None,
                           events=(None, None, None, None), stream=None):
    """Decode with torch.cuda.Event objects (enable_timing=True) recorded
    before/between/after the three kernels."""
    lib = load_library()
    ev = (ctypes.c_void_p * 4)(*[None if e is None else e.cuda_event for e in events])
    ro = ctypes.byref(route_out) if route_out is not None else None
    nbytes = scratch.numel() * scratch.element_size()
    _check(lib.si_debug_decode_events(plan.handle, ctypes.byref(layer), _ptr(x), int(n_tokens), _ptr(out),
                                      ro, _ptr(scratch), nbytes, ev, _stream(stream)),
           "si_debug_decode_events")


def si_debug_prefill_events(plan, layer: si_moe_layer, x, n_tokens, out, route_out=None, scratch=None,
                            events=(None, None, None, None, None), stream=None):
    """Prefill with torch.cuda.Event objects recorded before routing, before
    each GEMM, before the combine and after it."""
    lib = load_library()
    ev = (ctypes.c_void_p * 5)(*[None if e is None else e.cuda_event for e in events])
    ro = ctypes.byref(route_out) if route_out is not None else None
    nbytes = scratch.numel() * scratch.element_size()
    _check(lib.si_debug_prefill_events(plan.handle, ctypes.byref(layer), _ptr(x), int(n_tokens), _ptr(out),
                                       ro, _ptr(scratch), nbytes, ev, _stream(stream)),
           "si_debug_prefill_events")


def si_debug_plan_info(plan: Plan) -> dict:
    buf = (ctypes.c_int32 * 6)()
    load_library().si_debug_plan_info(plan.handle, buf, 6)
    keys = ("sm_count", "cluster_ok", "cluster_size", "clusters_resident", "clusters_needed", "smem_optin")
    return dict(zip(keys, list(buf)))


def si_debug_decode_fused(plan: Plan, n_tokens: int) -> int:
    return load_library().si_debug_decode_fused(plan.handle, int(n_tokens))


def si_moe_read_status(plan: Plan, scratch, stream=None) -> int:
    return load_library().si_moe_read_status(plan.handle, _ptr(scratch), _stream(stream))


def si_debug_q4k_dequant(blocks, n_blocks, out_f32=None, out_bf16=None, stream=None):
    _check(load_library().si_debug_q4k_dequant(_ptr(blocks), int(n_blocks), _ptr(out_f32),
                                               _ptr(out_bf16), _stream(stream)), "si_debug_q4k_dequant")


def si_debug_q4k_dequant_f16(blocks, n_blocks, out_f16, gamma=None, stream=None):
    _check(load_library().si_debug_q4k_dequant_f16(_ptr(blocks), int(n_blocks), _ptr(gamma), _ptr(out_f16),
                                                   _stream(stream)), "si_debug_q4k_dequant_f16")


def si_debug_nvfp4_dequant_f16(blocks, n_blocks, g, out_f16, stream=None):
    _check(load_library().si_debug_nvfp4_dequant_f16(_ptr(blocks), int(n_blocks), float(g), _ptr(out_f16),
                                                     _stream(stream)), "si_debug_nvfp4_dequant_f16")


def si_debug_q5k_dequant_f16(blocks, n_blocks, gamma, out_f16, stream=None):
    _check(load_library().si_debug_q5k_dequant_f16(_ptr(blocks), int(n_blocks), _ptr(gamma), _ptr(out_f16),
                                                   _stream(stream)), "si_debug_q5k_dequant_f16")


def si_moe_read_status_noalloc(stream=None) -> int:
    return load_library().si_moe_read_status_noalloc(_stream(stream))


def si_debug_topk(logits, n, desc: si_moe_desc, route_out: si_moe_route_out, stream=None):
    _check(load_library().si_debug_topk(_ptr(logits), int(n), ctypes.byref(desc),
                                        ctypes.byref(route_out), _stream(stream)), "si_debug_topk")
