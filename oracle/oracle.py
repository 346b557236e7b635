"""ctypes wrapper and build step for the C oracle (test infrastructure only).

The C source (oracle.c) is compiled with the host gcc into
oracle/_build/liboracle.so on first use, on whichever machine runs it.
No flags tune it for a particular CPU.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_DIR = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_DIR, "oracle.c")
_BUILD = os.path.join(_DIR, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_c_u8p = ctypes.POINTER(ctypes.c_uint8)
_c_u16p = ctypes.POINTER(ctypes.c_uint16)
_c_i32p = ctypes.POINTER(ctypes.c_int32)
_c_f32p = ctypes.POINTER(ctypes.c_float)
_c_f64p = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (plain -O2, no CPU-specific flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"],
                       check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.or_half_to_double.restype = ctypes.c_double
            lib.or_half_to_double.argtypes = [ctypes.c_uint16]
            lib.or_bf16_to_double.restype = ctypes.c_double
            lib.or_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.or_q4k_scale_min.argtypes = [_c_u8p, ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                             ctypes.POINTER(ctypes.c_int)]
            lib.or_q4k_dequant.argtypes = [_c_u8p, ctypes.c_int64, _c_f32p]
            lib.or_e2m1_to_double.restype = ctypes.c_double
            lib.or_e2m1_to_double.argtypes = [ctypes.c_int]
            lib.or_e4m3_to_double.restype = ctypes.c_double
            lib.or_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.or_nvfp4_dequant.argtypes = [_c_u8p, ctypes.c_int64, ctypes.c_float, _c_f32p]
            lib.or_q5k_dequant.argtypes = [_c_u8p, ctypes.c_int64, _c_f32p]
            lib.or_expert_ffn_wt.argtypes = [ctypes.c_int, _c_u8p, _c_u8p, _c_u8p, ctypes.c_float, ctypes.c_float,
                                             ctypes.c_float, ctypes.c_int, ctypes.c_int, _c_f64p, _c_f64p, _c_f64p]
            lib.or_moe_token_wt.argtypes = [ctypes.c_int, _c_u8p, _c_u8p, _c_u8p, _c_f32p, _c_f32p, _c_f32p,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _c_u16p,
                                            _c_i32p, _c_f64p, _c_f32p, _c_f64p, _c_f64p]
            lib.or_router_logits.argtypes = [_c_f32p, _c_f32p, _c_u16p, ctypes.c_int, ctypes.c_int,
                                             _c_f64p]
            lib.or_topk.argtypes = [_c_f32p, ctypes.c_int, ctypes.c_int, _c_i32p]
            lib.or_renorm_weights.argtypes = [_c_f64p, ctypes.c_int, _c_i32p, ctypes.c_int, _c_f64p]
            lib.or_route_tokens.argtypes = [_c_f32p, _c_f32p, _c_u16p, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, _c_i32p, _c_f64p, _c_f64p,
                                            _c_f64p]
            lib.or_expert_ffn.argtypes = [_c_u8p, _c_u8p, _c_u8p, ctypes.c_int, ctypes.c_int,
                                          _c_f64p, _c_f64p, _c_f64p]
            lib.or_moe_token.argtypes = [_c_u8p, _c_u8p, _c_u8p, _c_f32p, _c_f32p, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, _c_u16p, _c_i32p,
                                         _c_f64p, _c_f32p, _c_f64p, _c_f64p]
            lib.or_rmsnorm.argtypes = [_c_u16p, _c_f32p, ctypes.c_float, ctypes.c_int, _c_f64p]
            lib.or_route_tokens_prenorm.argtypes = [_c_f32p, _c_f32p, _c_f32p, ctypes.c_float, _c_u16p,
                                                    ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                    _c_i32p, _c_f64p, _c_f64p, _c_f64p]
            lib.or_moe_token_prenorm.argtypes = [_c_u8p, _c_u8p, _c_u8p, _c_f32p, _c_f32p, _c_f32p,
                                                 ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_int, _c_u16p, _c_i32p, _c_f64p, _c_f32p,
                                                 _c_f64p, _c_f64p]
            lib.or_counts_offsets_perm.argtypes = [_c_i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                   _c_i32p, _c_i32p, _c_i32p]
            _c_i8p = ctypes.POINTER(ctypes.c_int8)
            lib.or_act8_quant.argtypes = [_c_f32p, ctypes.c_int, _c_i8p, _c_f32p, _c_f64p]
            lib.or_expert_ffn_act8.argtypes = [_c_u8p, _c_u8p, _c_u8p, ctypes.c_int, ctypes.c_int, _c_f64p,
                                               _c_f64p, _c_f64p]
            lib.or_moe_token_act8.argtypes = [_c_u8p, _c_u8p, _c_u8p, _c_f32p, _c_f32p, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, _c_u16p, _c_i32p, _c_f64p, _c_f64p]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None, ctype):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctype)


def half_to_double(h: int) -> float:
    return _load().or_half_to_double(h)


def bf16_to_double(b: int) -> float:
    return _load().or_bf16_to_double(b)


def q4k_scale_min(scales12: np.ndarray, j: int) -> tuple[int, int]:
    s = np.ascontiguousarray(scales12, dtype=np.uint8)
    assert s.size == 12
    sc, m = ctypes.c_int(), ctypes.c_int()
    _load().or_q4k_scale_min(_ptr(s, _c_u8p), j, ctypes.byref(sc), ctypes.byref(m))
    return sc.value, m.value


def q4k_dequant(blocks: np.ndarray) -> np.ndarray:
    """fp32 weights of Q4_K blocks: any uint8 array whose size is a multiple of 144."""
    b = np.ascontiguousarray(blocks, dtype=np.uint8)
    n = b.size // 144
    assert n * 144 == b.size
    out = np.empty(n * 256, dtype=np.float32)
    _load().or_q4k_dequant(_ptr(b, _c_u8p), n, _ptr(out, _c_f32p))
    return out


WTYPE_Q4_K = 12
WTYPE_Q5_K = 13
WTYPE_NVFP4 = 100


def q5k_dequant(blocks: np.ndarray) -> np.ndarray:
    """fp32 weights of Q5_K blocks: any uint8 array whose size is a multiple of 176."""
    b = np.ascontiguousarray(blocks, dtype=np.uint8)
    n = b.size // 176
    assert n * 176 == b.size
    out = np.empty(n * 256, dtype=np.float32)
    _load().or_q5k_dequant(_ptr(b, _c_u8p), n, _ptr(out, _c_f32p))
    return out


def e2m1_to_double(code: int) -> float:
    return _load().or_e2m1_to_double(int(code))


def e4m3_to_double(b: int) -> float:
    return _load().or_e4m3_to_double(int(b))


def nvfp4_dequant(blocks: np.ndarray, g: float) -> np.ndarray:
    """fp32 weights of NVFP4 super-blocks (144 bytes per 256 weights) with tensor scale g."""
    b = np.ascontiguousarray(blocks, dtype=np.uint8)
    n = b.size // 144
    assert n * 144 == b.size
    out = np.empty(n * 256, dtype=np.float32)
    _load().or_nvfp4_dequant(_ptr(b, _c_u8p), n, float(np.float32(g)), _ptr(out, _c_f32p))
    return out


def router_logits(router_w: np.ndarray, x_bf16: np.ndarray, bias: np.ndarray | None = None):
    w = np.ascontiguousarray(router_w, dtype=np.float32)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    E, H = w.shape
    z = np.empty(E, dtype=np.float64)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    _load().or_router_logits(_ptr(w, _c_f32p), _ptr(b, _c_f32p), _ptr(x, _c_u16p), E, H,
                             _ptr(z, _c_f64p))
    return z


def topk(z32: np.ndarray, k: int) -> np.ndarray:
    z = np.ascontiguousarray(z32, dtype=np.float32)
    ids = np.empty(k, dtype=np.int32)
    _load().or_topk(_ptr(z, _c_f32p), z.size, k, _ptr(ids, _c_i32p))
    return ids


def renorm_weights(z: np.ndarray, ids: np.ndarray) -> np.ndarray:
    zz = np.ascontiguousarray(z, dtype=np.float64)
    ii = np.ascontiguousarray(ids, dtype=np.int32)
    w = np.empty(ii.size, dtype=np.float64)
    _load().or_renorm_weights(_ptr(zz, _c_f64p), zz.size, _ptr(ii, _c_i32p), ii.size,
                              _ptr(w, _c_f64p))
    return w


def route_tokens(router_w, x_bf16, k, bias=None, want_logits=False):
    """Route [T, H] tokens.  Returns (ids [T,k] i32, w [T,k] f64, z [T,E] f64|None, margin [T])."""
    w_r = np.ascontiguousarray(router_w, dtype=np.float32)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    E, H = w_r.shape
    T = x.shape[0]
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    z = np.empty((T, E), dtype=np.float64) if want_logits else None
    margin = np.empty(T, dtype=np.float64)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    _load().or_route_tokens(_ptr(w_r, _c_f32p), _ptr(b, _c_f32p), _ptr(x, _c_u16p), T, E, H, k,
                            _ptr(ids, _c_i32p), _ptr(w, _c_f64p), _ptr(z, _c_f64p),
                            _ptr(margin, _c_f64p))
    return ids, w, z, margin


def expert_ffn(wg_e, wu_e, wd_e, x64, H, I, wtype=WTYPE_Q4_K, gscales=(0.0, 0.0, 0.0)):
    """One expert's SwiGLU FFN in fp64 (Q4_K, or NVFP4 with the three matrices'
    tensor scales).  Returns (h [I], y [H])."""
    g = np.ascontiguousarray(wg_e, dtype=np.uint8)
    u = np.ascontiguousarray(wu_e, dtype=np.uint8)
    d = np.ascontiguousarray(wd_e, dtype=np.uint8)
    x = np.ascontiguousarray(x64, dtype=np.float64)
    h = np.empty(I, dtype=np.float64)
    y = np.empty(H, dtype=np.float64)
    gg, gu, gd = (float(np.float32(v)) for v in gscales)
    _load().or_expert_ffn_wt(int(wtype), _ptr(g, _c_u8p), _ptr(u, _c_u8p), _ptr(d, _c_u8p), gg, gu, gd, H, I,
                             _ptr(x, _c_f64p), _ptr(h, _c_f64p), _ptr(y, _c_f64p))
    return h, y


class TokenResult:
    __slots__ = ("ids", "w", "out32", "out64", "h")

    def __init__(self, ids, w, out32, out64, h):
        self.ids, self.w, self.out32, self.out64, self.h = ids, w, out32, out64, h


def moe_token(layer, x_bf16_row, want_h=False) -> TokenResult:
    """The MoE FFN for one token of a synth.MoeLayer-like object."""
    s = layer.shape
    H, I, E, k = s.hidden, s.intermediate, s.n_experts, s.top_k
    x = np.ascontiguousarray(x_bf16_row, dtype=np.uint16)
    assert x.size == H
    ids = np.empty(k, dtype=np.int32)
    w = np.empty(k, dtype=np.float64)
    out32 = np.empty(H, dtype=np.float32)
    out64 = np.empty(H, dtype=np.float64)
    h = np.empty((k, I), dtype=np.float64) if want_h else None
    bias = None if layer.router_bias is None else np.ascontiguousarray(layer.router_bias,
                                                                       dtype=np.float32)
    wtype = getattr(layer, "wtype", WTYPE_Q4_K)
    gsc = None
    if wtype == WTYPE_NVFP4:
        gsc = np.ascontiguousarray(layer.gscale, dtype=np.float32)
        assert gsc.shape == (E, 3)
    _load().or_moe_token_wt(int(wtype), _ptr(layer.w_gate, _c_u8p), _ptr(layer.w_up, _c_u8p),
                            _ptr(layer.w_down, _c_u8p), _ptr(gsc, _c_f32p), _ptr(layer.router_w, _c_f32p),
                            _ptr(bias, _c_f32p), H, I, E, k, _ptr(x, _c_u16p), _ptr(ids, _c_i32p),
                            _ptr(w, _c_f64p), _ptr(out32, _c_f32p), _ptr(out64, _c_f64p),
                            _ptr(h, _c_f64p))
    return TokenResult(ids, w, out32, out64, h)


def rmsnorm(x_bf16_row, gamma, eps: float) -> np.ndarray:
    """fp64 x * gamma / sqrt(mean(x^2) + eps) of one bf16 row."""
    x = np.ascontiguousarray(x_bf16_row, dtype=np.uint16)
    g = np.ascontiguousarray(gamma, dtype=np.float32)
    assert g.size == x.size
    xn = np.empty(x.size, dtype=np.float64)
    _load().or_rmsnorm(_ptr(x, _c_u16p), _ptr(g, _c_f32p), float(eps), x.size, _ptr(xn, _c_f64p))
    return xn


def route_tokens_prenorm(router_w, x_bf16, k, gamma, eps, bias=None):
    """Routing of [T, H] tokens of a pre-normed block: (ids, w, z [T,E] f64, margin [T])."""
    w_r = np.ascontiguousarray(router_w, dtype=np.float32)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    g = np.ascontiguousarray(gamma, dtype=np.float32)
    E, H = w_r.shape
    T = x.shape[0]
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    z = np.empty((T, E), dtype=np.float64)
    margin = np.empty(T, dtype=np.float64)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    _load().or_route_tokens_prenorm(_ptr(w_r, _c_f32p), _ptr(b, _c_f32p), _ptr(g, _c_f32p), float(eps),
                                    _ptr(x, _c_u16p), T, E, H, k, _ptr(ids, _c_i32p), _ptr(w, _c_f64p),
                                    _ptr(z, _c_f64p), _ptr(margin, _c_f64p))
    return ids, w, z, margin


class PrenormResult:
    __slots__ = ("ids", "w", "out32", "out64", "z")

    def __init__(self, ids, w, out32, out64, z):
        self.ids, self.w, self.out32, self.out64, self.z = ids, w, out32, out64, z

    @property
    def margin(self) -> float:
        """z_(k) - z_(k+1) of the sorted fp64 logits (+inf when k == E)."""
        k = self.ids.size
        if k >= self.z.size:
            return float("inf")
        zs = np.sort(self.z)[::-1]
        return float(zs[k - 1] - zs[k])


def moe_token_prenorm(layer, x_bf16_row, gamma, eps: float) -> PrenormResult:
    """out = x + MoE(rmsnorm(x)) for one token of a synth.MoeLayer-like object."""
    s = layer.shape
    H, I, E, k = s.hidden, s.intermediate, s.n_experts, s.top_k
    x = np.ascontiguousarray(x_bf16_row, dtype=np.uint16)
    g = np.ascontiguousarray(gamma, dtype=np.float32)
    assert x.size == H and g.size == H
    ids = np.empty(k, dtype=np.int32)
    w = np.empty(k, dtype=np.float64)
    out32 = np.empty(H, dtype=np.float32)
    out64 = np.empty(H, dtype=np.float64)
    z = np.empty(E, dtype=np.float64)
    bias = None if layer.router_bias is None else np.ascontiguousarray(layer.router_bias,
                                                                       dtype=np.float32)
    _load().or_moe_token_prenorm(_ptr(layer.w_gate, _c_u8p), _ptr(layer.w_up, _c_u8p),
                                 _ptr(layer.w_down, _c_u8p), _ptr(layer.router_w, _c_f32p),
                                 _ptr(bias, _c_f32p), _ptr(g, _c_f32p), float(eps), H, I, E, k,
                                 _ptr(x, _c_u16p), _ptr(ids, _c_i32p), _ptr(w, _c_f64p),
                                 _ptr(out32, _c_f32p), _ptr(out64, _c_f64p), _ptr(z, _c_f64p))
    return PrenormResult(ids, w, out32, out64, z)


def counts_offsets_perm(ids: np.ndarray, n_experts: int):
    """Prefill bookkeeping for ids [T, k]: (counts [E], offsets [E+1], perm [T*k])."""
    ii = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ii.shape
    counts = np.empty(n_experts, dtype=np.int32)
    offsets = np.empty(n_experts + 1, dtype=np.int32)
    perm = np.empty(T * k, dtype=np.int32)
    _load().or_counts_offsets_perm(_ptr(ii, _c_i32p), T, k, n_experts, _ptr(counts, _c_i32p),
                                   _ptr(offsets, _c_i32p), _ptr(perm, _c_i32p))
    return counts, offsets, perm


__all__ = [
    "build", "half_to_double", "bf16_to_double", "q4k_scale_min", "q4k_dequant",
    "WTYPE_Q4_K", "WTYPE_Q5_K", "q5k_dequant", "WTYPE_NVFP4", "e2m1_to_double", "e4m3_to_double", "nvfp4_dequant",
    "router_logits", "topk", "renorm_weights", "route_tokens", "expert_ffn", "moe_token",
    "TokenResult", "counts_offsets_perm", "rmsnorm", "moe_token_prenorm", "PrenormResult", "route_tokens_prenorm",
    "act8_quant", "expert_ffn_act8", "moe_token_act8",
]


# ----------------------------------------------------------------- int8-activation mode
def act8_quant(v32: np.ndarray):
    """Quantise fp32 values (a multiple of 32 of them) per 32-value block:
    (q int8 [n], d fp32 [n/32], s fp64 [n/32]) -- see oracle.c, int8-activation mode."""
    v = np.ascontiguousarray(v32, dtype=np.float32)
    n = v.size
    assert n % 32 == 0
    q = np.empty(n, dtype=np.int8)
    d = np.empty(n // 32, dtype=np.float32)
    s = np.empty(n // 32, dtype=np.float64)
    _load().or_act8_quant(_ptr(v, _c_f32p), n, q.ctypes.data_as(ctypes.POINTER(ctypes.c_int8)), _ptr(d, _c_f32p),
                          _ptr(s, _c_f64p))
    return q, d, s


def expert_ffn_act8(wg_e, wu_e, wd_e, x64, H, I):
    """One Q4_K expert's FFN in the int8-activation mode: (h [I], y [H]) in fp64."""
    g = np.ascontiguousarray(wg_e, dtype=np.uint8)
    u = np.ascontiguousarray(wu_e, dtype=np.uint8)
    d = np.ascontiguousarray(wd_e, dtype=np.uint8)
    x = np.ascontiguousarray(x64, dtype=np.float64)
    h = np.empty(I, dtype=np.float64)
    y = np.empty(H, dtype=np.float64)
    _load().or_expert_ffn_act8(_ptr(g, _c_u8p), _ptr(u, _c_u8p), _ptr(d, _c_u8p), H, I, _ptr(x, _c_f64p),
                               _ptr(h, _c_f64p), _ptr(y, _c_f64p))
    return h, y


def moe_token_act8(layer, x_bf16_row):
    """The MoE FFN of one token in the int8-activation mode (Q4_K layers): (ids, w, out64)."""
    s = layer.shape
    H, I, E, k = s.hidden, s.intermediate, s.n_experts, s.top_k
    x = np.ascontiguousarray(x_bf16_row, dtype=np.uint16)
    ids = np.empty(k, dtype=np.int32)
    w = np.empty(k, dtype=np.float64)
    out64 = np.empty(H, dtype=np.float64)
    bias = None if layer.router_bias is None else np.ascontiguousarray(layer.router_bias, dtype=np.float32)
    _load().or_moe_token_act8(_ptr(layer.w_gate, _c_u8p), _ptr(layer.w_up, _c_u8p), _ptr(layer.w_down, _c_u8p),
                              _ptr(layer.router_w, _c_f32p), _ptr(bias, _c_f32p), H, I, E, k, _ptr(x, _c_u16p),
                              _ptr(ids, _c_i32p), _ptr(w, _c_f64p), _ptr(out64, _c_f64p))
    return ids, w, out64
