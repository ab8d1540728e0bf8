"""Backward step of FP4 quantisation-aware training for the MoE layer's expert
path: plain numpy in float64 on top of the C oracle's codecs.

TEST INFRASTRUCTURE ONLY, like the rest of this package: the tests and
nothing else use it; it shares no code with the CUDA library.

What it follows ("DeepSeek-V4揭秘…" section 4, FP4 quantisation-aware
training): FP32 master weights are quantised to FP4 and dequantised to FP8
for compute; the backward computes with those FP8 weights and hands the
gradients to the master weights unchanged (a straight-through estimator for
the weight quantisation, with no re-quantisation of the transposed weights).
Section 3.2 (determinism): the MoE backward accumulates in a fixed token order.

Readings taken where the pages are silent, marked [R]:
  - Routing is held fixed: the gradient stops at the routing weights (dw is
    returned for a router backward) and does not flow through the gate. [R]
  - The FP8 quantisations of x and h in the forward are straight-through:
    the gradient with respect to a dequantised value passes to the value. [R]
  - The backward GEMMs read FP8 operands like the forward's: with
    quantize_grads, dy and [dg, du] are quantised to E4M3 per 128 channels
    with the activations' power-of-two rule before the GEMMs that read them
    (dh = W2^T dy, dx = W13^T [dg; du], and the two weight gradients). [R]
  - The SwiGLU backward uses the forward's g and u as rounded to fp32. [R]
  - Weight gradients sum over the expert's pairs in token order, then slot
    order; dx sums a token's slots in slot order. [R]
"""
import numpy as np

from . import bf16_to_f32, e4m3_decode, e4m3_encode, e4m3_scale_exp, expert_pair, fp4_to_fp8t, quant_act

_E4M3 = np.array([e4m3_decode(c) for c in range(256)], np.float64)


def fp8_weights(w_fp4, w_scale):
    """The FP8 weights the backward computes with, as float64 W [E, N, K]: the
    codes and 128x128 block exponents of fp4_to_fp8t, untransposed."""
    w8t, s8t = fp4_to_fp8t(w_fp4, w_scale)
    B = np.repeat(np.repeat(s8t.astype(np.int64) - 127, 128, axis=1), 128, axis=2)
    return (_E4M3[w8t] * np.ldexp(1.0, B)).transpose(0, 2, 1)


def fp4_weights(w_fp4, w_scale):
    """The forward's weights as float64 W [E, N, K] (E2M1 code * 2^scale)."""
    e2m1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])
    codes = np.stack([w_fp4 & 15, w_fp4 >> 4], axis=-1).reshape(*w_fp4.shape[:-1], -1)
    X = np.repeat(w_scale.astype(np.int64) - 127, 32, axis=-1)
    return e2m1[codes] * np.ldexp(1.0, X)


def q8(v):
    """Dequantised E4M3 of a float64 vector, per 128 channels, with the
    activations' rule: the smallest power-of-two scale 2^e with amax <= 448 * 2^e."""
    out = np.empty_like(v)
    for g in range(v.shape[0] // 128):
        blk = v[g * 128:(g + 1) * 128]
        e = e4m3_scale_exp(float(np.abs(blk).max()))
        codes = [e4m3_encode(float(np.ldexp(x, -e))) for x in blk]
        out[g * 128:(g + 1) * 128] = _E4M3[codes] * np.ldexp(1.0, e)
    return out


def pair_dgu(g, u, dy, W2e, quantize_grads=True):
    """The first half of one token-expert pair's backward, from the gradient
    at y: dh = W2^T dy (on the FP8 weights), then the SwiGLU backward
    dg = dh u sig(g) (1 + g (1 - sig(g))), du = dh g sig(g).  g, u are the
    forward's (rounded to fp32), dy the pair's gradient at y (w_j dout).
    Returns (dyq, dg, du, dgu): dy as the GEMM reads it (E4M3 per 128 channels
    with quantize_grads), dg and du unquantised, and [dg; du] as the next
    GEMM reads it (E4M3 per 128 channels with quantize_grads)."""
    if quantize_grads:
        dy = q8(dy)
    dh = W2e.T @ dy
    sig = 1.0 / (1.0 + np.exp(-g))
    dg = dh * u * sig * (1.0 + g * (1.0 - sig))
    du = dh * g * sig
    dgu = np.concatenate([dg, du])
    if quantize_grads:
        dgu = q8(dgu)
    return dy, dg, du, dgu


def forward_gu(xq_row, xs_row, e, w13_fp4, w13_scale):
    """g and u of a pair as the forward computes them: exact sums rounded to fp32."""
    xd = _E4M3[xq_row] * np.ldexp(1.0, np.repeat(np.asarray(xs_row, np.int64) - 127, 128))
    W13f = fp4_weights(w13_fp4[e:e + 1], w13_scale[e:e + 1])[0]
    inter = W13f.shape[0] // 2
    g = (W13f[:inter] @ xd).astype(np.float32).astype(np.float64)
    u = (W13f[inter:] @ xd).astype(np.float32).astype(np.float64)
    return g, u


def qat_backward(x, topk_idx, topk_w, w13_fp4, w13_scale, w2_fp4, w2_scale, dout, quantize_grads=True):
    """Gradients of the layer output's inner product with `dout` (bf16 bits
    [T, d]) for the forward of x (bf16 bits [T, d]) under the given routing.

    Returns (dx [T, d], dw [T, k], dW13 [E, 2I, d], dW2 [E, d, I]), float64:
    dx through the experts, dw with respect to the routing weights, and the
    master weights' gradients.
    """
    x = np.asarray(x, np.uint16)
    T, d = x.shape
    k = topk_idx.shape[1]
    xq, xs = quant_act(x)
    xd = _E4M3[xq] * np.ldexp(1.0, np.repeat(xs.astype(np.int64) - 127, 128, axis=1))
    W13f = fp4_weights(w13_fp4, w13_scale)                 # the forward's weights (g, u)
    W13 = fp8_weights(w13_fp4, w13_scale)                  # the backward's
    W2 = fp8_weights(w2_fp4, w2_scale)
    E, twoI, _ = W13.shape
    inter = twoI // 2
    do = np.array([[bf16_to_f32(b) for b in row] for row in np.asarray(dout, np.uint16)], np.float64)
    dx = np.zeros((T, d))
    dw = np.zeros((T, k))
    dW13 = np.zeros((E, twoI, d))
    dW2 = np.zeros((E, d, inter))
    for t in range(T):
        for j in range(k):
            e = int(topk_idx[t, j])
            g = (W13f[e, :inter] @ xd[t]).astype(np.float32).astype(np.float64)
            u = (W13f[e, inter:] @ xd[t]).astype(np.float32).astype(np.float64)
            _, hq, hs, y = expert_pair(xq[t], xs[t], e, w13_fp4, w13_scale, w2_fp4, w2_scale)
            yf = np.array([bf16_to_f32(b) for b in y], np.float64)
            hd = _E4M3[hq] * np.ldexp(1.0, np.repeat(hs.astype(np.int64) - 127, 128))
            dy = float(topk_w[t, j]) * do[t]
            dw[t, j] = do[t] @ yf
            dy, _, _, dgu = pair_dgu(g, u, dy, W2[e], quantize_grads)
            dx[t] += W13[e].T @ dgu
            dW2[e] += np.outer(dy, hd)
            dW13[e] += np.outer(dgu, xd[t])
    return dx, dw, dW13, dW2
