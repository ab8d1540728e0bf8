"""Thin ctypes binding of libfp4moe.so (include/fp4moe.h), same names.

Argument marshalling only: torch tensors become device pointers and the current
torch stream becomes the cudaStream_t; every step of the layer runs in the
library's CUDA kernels.  If the library has not been built, importing this
module raises -- there is no other implementation to fall back to.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libfp4moe.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("libfp4moe.so is not built (%s); run fp4_expert_grouped_gb300/build.py "
                      "or __graft_entry__.build()" % LIB_PATH)

_lib = ctypes.CDLL(LIB_PATH)

MOE_OK = 0
STATUS_NAMES = {
    0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED_SHAPE", 3: "MOE_ERR_CUDA",
    4: "MOE_ERR_WORKSPACE", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_UNSUPPORTED_DEVICE", 7: "MOE_ERR_DEVICE_FAULT",
}
STAGES = ["gate", "topk", "plan", "dispatch", "gemm1", "gemm2", "combine"]
(MOE_WS_XQ, MOE_WS_XS, MOE_WS_LOGITS, MOE_WS_TOPK_IDX, MOE_WS_TOPK_W, MOE_WS_EXPERT_OFFSETS,
 MOE_WS_SORTED_PAIR, MOE_WS_PAIR_POS, MOE_WS_TILE_PREFIX, MOE_WS_HQ, MOE_WS_HS_TILES, MOE_WS_Y,
 MOE_WS_XQ_SORTED, MOE_WS_XS_TILES, MOE_WS_PLAN_COUNTS, MOE_WS_TILE_DONE, MOE_WS_TOPK_Z, MOE_WS_GATE_WT,
 MOE_WS_GATE_WHI, MOE_WS_GATE_WLO, MOE_WS_GATE_WNORM, MOE_WS_GATE_NCAND, MOE_WS_COUNT) = range(23)
# from this many tokens (E a multiple of 64) the gate runs on the tensor cores
# with certified routing (include/fp4moe.h)
MOE_GATE_TC_MIN_TOKENS = 1024

# every symbol the header declares
EXPORTS = ["moe_status_string", "moe_version", "moe_pack_fp4", "moe_fp4_to_fp8t", "moe_quantize_act", "moe_route",
           "moe_route_noalloc", "moe_dispatch_plan", "moe_forward", "moe_forward_ex", "moe_workspace_size",
           "moe_workspace_layout", "moe_get_device_status", "moe_backward_h", "moe_backward_h_workspace_size",
           "moe_backward_x", "moe_backward_x_workspace_size", "moe_backward_dw",
           "moe_backward_w", "moe_backward_w_workspace_size", "moe_gate_prep_size", "moe_prepare_gate"]


class MoeForwardOpts(ctypes.Structure):
    _fields_ = [("gate_bias", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("topk_idx_out", ctypes.c_void_p),
                ("topk_w_out", ctypes.c_void_p), ("pair_pos_out", ctypes.c_void_p),
                ("flags", ctypes.c_uint32), ("stage_events", ctypes.POINTER(ctypes.c_void_p)),
                ("gu_out", ctypes.c_void_p), ("gate_prep", ctypes.c_void_p)]


_vp, _i, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_lib.moe_status_string.argtypes = [_i]
_lib.moe_status_string.restype = ctypes.c_char_p
_lib.moe_version.argtypes = []
_lib.moe_version.restype = _i
_lib.moe_pack_fp4.argtypes = [_vp, _vp, _vp, _i, _i, _i, _vp]
_lib.moe_pack_fp4.restype = _i
_lib.moe_fp4_to_fp8t.argtypes = [_vp, _vp, _vp, _vp, _i, _i, _i, _vp]
_lib.moe_fp4_to_fp8t.restype = _i
_lib.moe_quantize_act.argtypes = [_vp, _vp, _vp, _i, _i, _vp]
_lib.moe_quantize_act.restype = _i
_lib.moe_route.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp]
_lib.moe_route.restype = _i
_lib.moe_route_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp]
_lib.moe_route_noalloc.restype = _i
_lib.moe_dispatch_plan.argtypes = [_vp, _vp, _vp, _vp, _i, _i, _i, _vp]
_lib.moe_dispatch_plan.restype = _i
_lib.moe_forward.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]
_lib.moe_forward.restype = _i
_lib.moe_forward_ex.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp,
                                ctypes.POINTER(MoeForwardOpts)]
_lib.moe_forward_ex.restype = _i
_lib.moe_workspace_size.argtypes = [_i, _i, _i, _i, _i]
_lib.moe_workspace_size.restype = _sz
_lib.moe_workspace_layout.argtypes = [_i, _i, _i, _i, _i, ctypes.POINTER(_sz), ctypes.POINTER(_sz)]
_lib.moe_workspace_layout.restype = _sz
_lib.moe_get_device_status.argtypes = [_vp]
_lib.moe_get_device_status.restype = _i
_lib.moe_backward_h_workspace_size.argtypes = [_i, _i, _i, _i, _i]
_lib.moe_backward_h_workspace_size.restype = _sz
_lib.moe_backward_h.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]
_lib.moe_backward_h.restype = _i
_lib.moe_backward_x_workspace_size.argtypes = [_i, _i, _i, _i, _i]
_lib.moe_backward_x_workspace_size.restype = _sz
_lib.moe_backward_x.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _i, _i, _i, _i, _i, _vp]
_lib.moe_backward_x.restype = _i
_lib.moe_backward_dw.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]
_lib.moe_backward_dw.restype = _i
_lib.moe_backward_w_workspace_size.argtypes = [_i, _i, _i, _i, _i]
_lib.moe_backward_w_workspace_size.restype = _sz
_lib.moe_backward_w.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i, _i, _i, _i, _i, _vp]
_lib.moe_backward_w.restype = _i
_lib.moe_gate_prep_size.argtypes = [_i, _i]
_lib.moe_gate_prep_size.restype = _sz
_lib.moe_prepare_gate.argtypes = [_vp, _vp, _i, _i, _vp]
_lib.moe_prepare_gate.restype = _i


class MoeError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        super().__init__("%s failed: %s" % (what, STATUS_NAMES.get(code, code)))


def lib():
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code, what):
    if code != MOE_OK:
        raise MoeError(code, what)


def moe_status_string(code):
    return _lib.moe_status_string(code).decode()


def moe_version():
    return _lib.moe_version()


def moe_pack_fp4(w, w_fp4, w_scale, stream=None):
    """w fp32 [E, N, K] -> tiled MXFP4: w_fp4 (E*N*K/2 bytes), w_scale (E*N*K/32 bytes),
    device tensors of any shape with that many bytes (see include/fp4moe.h)."""
    E, N, K = w.shape if w.dim() == 3 else (1, *w.shape)
    _check(_lib.moe_pack_fp4(_ptr(w), _ptr(w_fp4), _ptr(w_scale), E, N, K, _stream(stream)), "moe_pack_fp4")


def moe_fp4_to_fp8t(w_fp4, w_scale, w8t, s8t, stream=None):
    """w_fp4 uint8 [E, N, K/2], w_scale [E, N, K/32] (moe_pack_fp4 output) ->
    w8t uint8 [E, K, N] bytes: E4M3 codes of W^T in the header's tiled block order,
    s8t uint8 [E, K/128, N/128] block exponents + 127."""
    E, N, K2 = w_fp4.shape
    _check(_lib.moe_fp4_to_fp8t(_ptr(w_fp4), _ptr(w_scale), _ptr(w8t), _ptr(s8t), E, N, 2 * K2, _stream(stream)),
           "moe_fp4_to_fp8t")


def moe_quantize_act(x, xq, xs, stream=None):
    T, d = x.shape
    _check(_lib.moe_quantize_act(_ptr(x), _ptr(xq), _ptr(xs), T, d, _stream(stream)), "moe_quantize_act")


def moe_route(x, gate_w, gate_bias, topk_idx, topk_w, stream=None):
    T, d = x.shape
    E = gate_w.shape[1]
    k = topk_idx.shape[1]
    _check(_lib.moe_route(_ptr(x), _ptr(gate_w), _ptr(gate_bias), _ptr(topk_idx), _ptr(topk_w),
                          T, d, E, k, _stream(stream)), "moe_route")


def moe_route_noalloc(x, gate_w, gate_bias, topk_idx, topk_w, stream=None):
    """moe_route whose logits scratch is the library's fixed device array
    (nothing is allocated; T * E <= 1048576; overlapping calls race)."""
    T, d = x.shape
    E = gate_w.shape[1]
    k = topk_idx.shape[1]
    _check(_lib.moe_route_noalloc(_ptr(x), _ptr(gate_w), _ptr(gate_bias), _ptr(topk_idx), _ptr(topk_w),
                                  T, d, E, k, _stream(stream)), "moe_route_noalloc")


def moe_dispatch_plan(topk_idx, expert_offsets, sorted_pair, pair_pos, E, stream=None):
    T, k = topk_idx.shape
    _check(_lib.moe_dispatch_plan(_ptr(topk_idx), _ptr(expert_offsets), _ptr(sorted_pair), _ptr(pair_pos),
                                  T, E, k, _stream(stream)), "moe_dispatch_plan")


def moe_workspace_size(T, d, inter, E, k):
    return _lib.moe_workspace_size(T, d, inter, E, k)


def moe_workspace_layout(T, d, inter, E, k):
    """Return (total_bytes, offsets[list], strides[list])."""
    off = (_sz * MOE_WS_COUNT)()
    st = (_sz * MOE_WS_COUNT)()
    total = _lib.moe_workspace_layout(T, d, inter, E, k, off, st)
    return total, list(off), list(st)


def moe_forward(x, gate_w, w13_fp4, w13_scale, w2_fp4, w2_scale, out, k, stream=None):
    T, d = x.shape
    E = gate_w.shape[1]
    inter = w13_fp4.shape[1] // 2
    _check(_lib.moe_forward(_ptr(x), _ptr(gate_w), _ptr(w13_fp4), _ptr(w13_scale), _ptr(w2_fp4),
                            _ptr(w2_scale), _ptr(out), T, d, inter, E, k, _stream(stream)), "moe_forward")


def moe_forward_ex(x, gate_w, w13_fp4, w13_scale, w2_fp4, w2_scale, out, k, stream=None, gate_bias=None,
                   workspace=None, topk_idx_out=None, topk_w_out=None, pair_pos_out=None, flags=0,
                   stage_events=None, gu_out=None, gate_prep=None):
    """stage_events: optional list of len(STAGES) + 1 recorded torch.cuda.Event objects."""
    T, d = x.shape
    E = gate_w.shape[1]
    inter = w13_fp4.shape[1] // 2
    evs = None
    if stage_events is not None:
        assert len(stage_events) == len(STAGES) + 1
        evs = (ctypes.c_void_p * len(stage_events))(*[ev.cuda_event for ev in stage_events])
    o = MoeForwardOpts(_ptr(gate_bias), _ptr(workspace),
                       0 if workspace is None else workspace.numel() * workspace.element_size(),
                       _ptr(topk_idx_out), _ptr(topk_w_out), _ptr(pair_pos_out), flags,
                       ctypes.cast(evs, ctypes.POINTER(ctypes.c_void_p)) if evs is not None else None,
                       _ptr(gu_out), _ptr(gate_prep))
    _check(_lib.moe_forward_ex(_ptr(x), _ptr(gate_w), _ptr(w13_fp4), _ptr(w13_scale), _ptr(w2_fp4),
                               _ptr(w2_scale), _ptr(out), T, d, inter, E, k, _stream(stream),
                               ctypes.byref(o)), "moe_forward_ex")


def moe_gate_prep_size(d, E):
    return _lib.moe_gate_prep_size(d, E)


def moe_prepare_gate(gate_w, prep, stream=None):
    """gate_w fp32 [d, E] -> prep (uint8, moe_gate_prep_size(d, E) bytes): the tensor-core gate's form of it."""
    d, E = gate_w.shape
    _check(_lib.moe_prepare_gate(_ptr(gate_w), _ptr(prep), d, E, _stream(stream)), "moe_prepare_gate")


def moe_backward_h_workspace_size(T, d, inter, E, k):
    return _lib.moe_backward_h_workspace_size(T, d, inter, E, k)


def moe_backward_h(dout, w2_fp8t, w2_s8t, gu, fwd_workspace, dgu, dgu_scale, k, dgu_f32=None, workspace=None,
                   stream=None):
    """dout bf16 [T, d], w2_fp8t uint8 [E, inter, d] + w2_s8t [E, inter/128, d/128] (moe_fp4_to_fp8t
    of W2), gu fp32 [T*k, 2*inter] (moe_forward_ex gu_out), fwd_workspace: that forward's workspace;
    outputs dgu uint8 [T*k, 2*inter] (E4M3), dgu_scale uint8 [T*k, 2*inter/128], optionally dgu_f32."""
    T, d = dout.shape
    E, inter, _ = w2_fp8t.shape
    _check(_lib.moe_backward_h(_ptr(dout), _ptr(w2_fp8t), _ptr(w2_s8t), _ptr(gu), _ptr(fwd_workspace),
                               _ptr(workspace), 0 if workspace is None else workspace.numel() * workspace.element_size(),
                               _ptr(dgu), _ptr(dgu_scale), _ptr(dgu_f32), T, d, inter, E, k, _stream(stream)),
           "moe_backward_h")


def moe_backward_x_workspace_size(T, d, inter, E, k):
    return _lib.moe_backward_x_workspace_size(T, d, inter, E, k)


def moe_backward_x(dgu, dgu_scale, w13_fp8t, w13_s8t, fwd_workspace, dx, k, workspace=None, stream=None):
    """dgu uint8 [T*k, 2*inter] + dgu_scale [T*k, 2*inter/128] (moe_backward_h outputs), w13_fp8t uint8
    [E, d, 2*inter] + w13_s8t [E, d/128, 2*inter/128] (moe_fp4_to_fp8t of W13), fwd_workspace: the
    forward's workspace; output dx bf16 [T, d]."""
    T, d = dx.shape
    E, _, twoI = w13_fp8t.shape
    _check(_lib.moe_backward_x(_ptr(dgu), _ptr(dgu_scale), _ptr(w13_fp8t), _ptr(w13_s8t), _ptr(fwd_workspace),
                               _ptr(workspace), 0 if workspace is None else workspace.numel() * workspace.element_size(),
                               _ptr(dx), T, d, twoI // 2, E, k, _stream(stream)),
           "moe_backward_x")


def moe_backward_dw(dout, fwd_workspace, dw, inter, E, stream=None):
    """dout bf16 [T, d], fwd_workspace: the forward's workspace; output dw fp32 [T, k]."""
    T, d = dout.shape
    k = dw.shape[1]
    _check(_lib.moe_backward_dw(_ptr(dout), _ptr(fwd_workspace), _ptr(dw), T, d, inter, E, k, _stream(stream)),
           "moe_backward_dw")


def moe_backward_w_workspace_size(T, d, inter, E, k):
    return _lib.moe_backward_w_workspace_size(T, d, inter, E, k)


def moe_backward_w(fwd_workspace, bwd_h_workspace, dgu, dgu_scale, dW13, dW2, k, workspace=None, stream=None):
    """fwd_workspace: the forward's workspace; bwd_h_workspace: the workspace moe_backward_h was given;
    dgu, dgu_scale: moe_backward_h's outputs; outputs dW13 fp32 [E, 2*inter, d], dW2 fp32 [E, d, inter]."""
    E, d, inter = dW2.shape
    T = dgu.shape[0] // k
    _check(_lib.moe_backward_w(_ptr(fwd_workspace), _ptr(bwd_h_workspace), _ptr(dgu), _ptr(dgu_scale), _ptr(dW13),
                               _ptr(dW2), _ptr(workspace),
                               0 if workspace is None else workspace.numel() * workspace.element_size(),
                               T, d, inter, E, k, _stream(stream)),
           "moe_backward_w")


def moe_get_device_status(stream=None):
    """Synchronise the stream and return (and clear) the device status code."""
    return _lib.moe_get_device_status(_stream(stream))
