"""ctypes wrapper around the plain C oracle (oracle/moe_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
benchmark's CPU-baseline leg may import this module.  It shares no code with
the CUDA library and never imports it.

All functions take and return numpy arrays:
  x        uint16 [T, d]          bf16 bit patterns
  gate_w   float32 [d, E]
  w        float32 [E, N, K]      weights to pack (N = 2*inter for W13, d for W2)
  w_fp4    uint8 [E, N, K/2]      two E2M1 codes per byte, low nibble = even K
  w_scale  uint8 [E, N, K/32]     UE8M0 (exponent + 127)
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load(path):
    L = ctypes.CDLL(path)
    u8p = ctypes.POINTER(ctypes.c_uint8)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    i32p = ctypes.POINTER(ctypes.c_int32)
    f32p = ctypes.POINTER(ctypes.c_float)
    c_int = ctypes.c_int
    L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
    L.orc_bf16_to_f32.restype = ctypes.c_float
    L.orc_f32_to_bf16.argtypes = [ctypes.c_float]
    L.orc_f32_to_bf16.restype = ctypes.c_uint16
    L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
    L.orc_e4m3_decode.restype = ctypes.c_double
    L.orc_e4m3_encode.argtypes = [ctypes.c_double]
    L.orc_e4m3_encode.restype = ctypes.c_uint8
    L.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
    L.orc_e2m1_decode.restype = ctypes.c_double
    L.orc_e2m1_encode.argtypes = [ctypes.c_double]
    L.orc_e2m1_encode.restype = ctypes.c_uint8
    L.orc_e4m3_scale_exp.argtypes = [ctypes.c_double]
    L.orc_e4m3_scale_exp.restype = c_int
    L.orc_mx_scale_exp.argtypes = [ctypes.c_double]
    L.orc_mx_scale_exp.restype = c_int
    L.orc_gate_score.argtypes = [ctypes.c_float]
    L.orc_gate_score.restype = ctypes.c_float
    L.orc_quant_act.argtypes = [u16p, c_int, c_int, u8p, u8p]
    L.orc_quant_act.restype = None
    L.orc_pack_fp4.argtypes = [f32p, c_int, c_int, c_int, u8p, u8p]
    L.orc_pack_fp4.restype = None
    L.orc_fp4_to_fp8t.argtypes = [u8p, u8p, c_int, c_int, c_int, u8p, u8p]
    L.orc_fp4_to_fp8t.restype = None
    L.orc_gate_logits.argtypes = [u16p, f32p, f32p, c_int, c_int, c_int, f32p]
    L.orc_gate_logits.restype = None
    L.orc_topk.argtypes = [f32p, c_int, c_int, c_int, i32p, f32p]
    L.orc_topk.restype = c_int
    L.orc_dispatch_plan.argtypes = [i32p, c_int, c_int, c_int, i32p, i32p, i32p]
    L.orc_dispatch_plan.restype = c_int
    L.orc_expert_pair.argtypes = [u8p, u8p, c_int, u8p, u8p, u8p, u8p, c_int, c_int,
                                  ctypes.POINTER(ctypes.c_double), f32p, u8p, u8p, u16p]
    L.orc_expert_pair.restype = None
    L.orc_moe_forward.argtypes = [u16p, f32p, f32p, u8p, u8p, u8p, u8p,
                                  c_int, c_int, c_int, c_int, c_int,
                                  i32p, c_int, u16p, i32p, f32p]
    L.orc_moe_forward.restype = c_int
    L.orc_num_threads.argtypes = []
    L.orc_num_threads.restype = c_int
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = _load(_build.build())
    return _lib


class use_library:
    """Context manager: route every oracle call through another build of the
    oracle (a variant with a planted mistake, built by build.build_source),
    then restore the normal library.  Used only by the tests that check that
    the pins catch such mistakes."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        global _lib
        self.saved = lib()
        _lib = _load(self.path)
        return _lib

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def _p(a, ctype):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- scalar codecs --------------------------------------------------------

def bf16_to_f32(b):
    return lib().orc_bf16_to_f32(int(b))


def f32_to_bf16(f):
    return lib().orc_f32_to_bf16(float(f))


def e4m3_decode(c):
    return lib().orc_e4m3_decode(int(c))


def e4m3_encode(v):
    return lib().orc_e4m3_encode(float(v))


def e2m1_decode(c):
    return lib().orc_e2m1_decode(int(c))


def e2m1_encode(v):
    return lib().orc_e2m1_encode(float(v))


def e4m3_scale_exp(amax):
    return lib().orc_e4m3_scale_exp(float(amax))


def mx_scale_exp(amax):
    return lib().orc_mx_scale_exp(float(amax))


def gate_score(z):
    return lib().orc_gate_score(float(z))


def num_threads():
    return lib().orc_num_threads()


# ---- array stages ---------------------------------------------------------

def quant_act(x):
    x = _c(x, np.uint16)
    T, d = x.shape
    xq = np.empty((T, d), np.uint8)
    xs = np.empty((T, d // 128), np.uint8)
    lib().orc_quant_act(_p(x, ctypes.c_uint16), T, d, _p(xq, ctypes.c_uint8), _p(xs, ctypes.c_uint8))
    return xq, xs


def pack_fp4(w):
    w = _c(w, np.float32)
    if w.ndim == 2:
        w = w[None]
    E, N, K = w.shape
    w_fp4 = np.empty((E, N, K // 2), np.uint8)
    w_scale = np.empty((E, N, K // 32), np.uint8)
    lib().orc_pack_fp4(_p(w, ctypes.c_float), E, N, K, _p(w_fp4, ctypes.c_uint8), _p(w_scale, ctypes.c_uint8))
    return w_fp4, w_scale


def fp4_to_fp8t(w_fp4, w_scale):
    """FP8 weights for the backward pass, transposed: (w8t uint8 [E, K, N]
    E4M3 codes, s8t uint8 [E, K/128, N/128] UE8M0 block exponents + 127)."""
    w_fp4 = _c(w_fp4, np.uint8)
    w_scale = _c(w_scale, np.uint8)
    if w_fp4.ndim == 2:
        w_fp4, w_scale = w_fp4[None], w_scale[None]
    E, N, K2 = w_fp4.shape
    K = 2 * K2
    w8t = np.empty((E, K, N), np.uint8)
    s8t = np.empty((E, K // 128, N // 128), np.uint8)
    lib().orc_fp4_to_fp8t(_p(w_fp4, ctypes.c_uint8), _p(w_scale, ctypes.c_uint8), E, N, K,
                          _p(w8t, ctypes.c_uint8), _p(s8t, ctypes.c_uint8))
    return w8t, s8t


def gate_logits(x, gate_w, bias=None):
    x = _c(x, np.uint16)
    gate_w = _c(gate_w, np.float32)
    T, d = x.shape
    E = gate_w.shape[1]
    z = np.empty((T, E), np.float32)
    b = None if bias is None else _c(bias, np.float32)
    lib().orc_gate_logits(_p(x, ctypes.c_uint16), _p(gate_w, ctypes.c_float),
                          _p(b, ctypes.c_float), T, d, E, _p(z, ctypes.c_float))
    return z


def topk(z, k):
    z = _c(z, np.float32)
    T, E = z.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    rc = lib().orc_topk(_p(z, ctypes.c_float), T, E, k, _p(idx, ctypes.c_int32), _p(w, ctypes.c_float))
    if rc != 0:
        raise ValueError("orc_topk failed (%d)" % rc)
    return idx, w


def route(x, gate_w, k, bias=None):
    return topk(gate_logits(x, gate_w, bias), k)


def dispatch_plan(idx, E):
    idx = _c(idx, np.int32)
    T, k = idx.shape
    offs = np.empty(E + 1, np.int32)
    sp = np.empty(T * k, np.int32)
    pp = np.empty(T * k, np.int32)
    rc = lib().orc_dispatch_plan(_p(idx, ctypes.c_int32), T, E, k, _p(offs, ctypes.c_int32),
                                 _p(sp, ctypes.c_int32), _p(pp, ctypes.c_int32))
    if rc != 0:
        raise ValueError("orc_dispatch_plan failed (%d)" % rc)
    return offs, sp, pp


def expert_pair(xq_row, xs_row, e, w13_fp4, w13_scale, w2_fp4, w2_scale):
    """One token-expert pair; returns (h fp32 [inter], hq, hs, y bf16 bits [d])."""
    xq_row = _c(xq_row, np.uint8)
    xs_row = _c(xs_row, np.uint8)
    w13_fp4 = _c(w13_fp4, np.uint8)
    w13_scale = _c(w13_scale, np.uint8)
    w2_fp4 = _c(w2_fp4, np.uint8)
    w2_scale = _c(w2_scale, np.uint8)
    d = xq_row.shape[0]
    inter = w13_fp4.shape[1] // 2
    scratch = np.empty(max(d, inter), np.float64)
    h = np.empty(inter, np.float32)
    hq = np.empty(inter, np.uint8)
    hs = np.empty(inter // 128, np.uint8)
    y = np.empty(d, np.uint16)
    lib().orc_expert_pair(_p(xq_row, ctypes.c_uint8), _p(xs_row, ctypes.c_uint8), int(e),
                          _p(w13_fp4, ctypes.c_uint8), _p(w13_scale, ctypes.c_uint8),
                          _p(w2_fp4, ctypes.c_uint8), _p(w2_scale, ctypes.c_uint8), d, inter,
                          _p(scratch, ctypes.c_double), _p(h, ctypes.c_float),
                          _p(hq, ctypes.c_uint8), _p(hs, ctypes.c_uint8), _p(y, ctypes.c_uint16))
    return h, hq, hs, y


def moe_forward(x, gate_w, w13_fp4, w13_scale, w2_fp4, w2_scale, k, bias=None, tokens=None):
    """Oracle layer forward.  Returns (out bf16 bits [n, d], topk_idx [n, k], topk_w [n, k])
    for the listed tokens (all tokens when tokens is None)."""
    x = _c(x, np.uint16)
    gate_w = _c(gate_w, np.float32)
    w13_fp4 = _c(w13_fp4, np.uint8)
    w13_scale = _c(w13_scale, np.uint8)
    w2_fp4 = _c(w2_fp4, np.uint8)
    w2_scale = _c(w2_scale, np.uint8)
    T, d = x.shape
    E = gate_w.shape[1]
    inter = w13_fp4.shape[1] // 2
    assert w13_fp4.shape == (E, 2 * inter, d // 2)
    assert w2_fp4.shape == (E, d, inter // 2)
    tok = None if tokens is None else _c(tokens, np.int32)
    n = T if tok is None else tok.shape[0]
    out = np.empty((n, d), np.uint16)
    idx = np.empty((n, k), np.int32)
    w = np.empty((n, k), np.float32)
    b = None if bias is None else _c(bias, np.float32)
    rc = lib().orc_moe_forward(_p(x, ctypes.c_uint16), _p(gate_w, ctypes.c_float), _p(b, ctypes.c_float),
                               _p(w13_fp4, ctypes.c_uint8), _p(w13_scale, ctypes.c_uint8),
                               _p(w2_fp4, ctypes.c_uint8), _p(w2_scale, ctypes.c_uint8),
                               T, d, inter, E, k, _p(tok, ctypes.c_int32), n,
                               _p(out, ctypes.c_uint16), _p(idx, ctypes.c_int32), _p(w, ctypes.c_float))
    if rc != 0:
        raise ValueError("orc_moe_forward failed (%d)" % rc)
    return out, idx, w
